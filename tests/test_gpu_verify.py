"""GPU parts of the verify block: token embedding from the tied readout, per-row
argmax, and greedy generation with prompt-lookup drafts, which must give exactly
the tokens of plain one-token greedy decoding (Husky page, the passage before
"Flash draft model and candidate selection": the text does not change)."""
import numpy as np
import pytest
import torch

import oracle
from parity import dev_bf16, pack
from skinny_gemm_bit_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    from skinny_gemm_bit_gb300 import build
    build.build()
    from skinny_gemm_bit_gb300 import tfq
    return tfq


def _bf16_rne(a: np.ndarray) -> np.ndarray:
    # fp64 values that are exact in fp32 (dequantised weights are), rounded to bf16
    return synth.f32_to_bf16_bits(a.astype(np.float32))


@pytest.mark.parametrize("bits", [4, 8])
def test_embed_rows_are_the_dequantised_rows_bit_exact(T, bits):
    rng = np.random.default_rng(700 + bits)
    N, K = 1000, 512  # ragged last row block
    w = synth.quant_weights(rng, N, K, bits)
    ids = np.array([0, 999, 17, 500, 999, 3], dtype=np.int32)
    ws = T.workspace(256)
    x = T.tf_embed_rows(pack(T, w), torch.from_numpy(ids).cuda(), ws=ws)
    expect = _bf16_rne(oracle.dequant(w)[ids])
    got = x.cpu().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, expect)
    assert T.tf_workspace_status(ws) == T.TF_OK


def test_embed_rows_reports_an_id_outside_the_matrix(T):
    rng = np.random.default_rng(710)
    w = synth.quant_weights(rng, 64, 128, 4)
    ws = T.workspace(256)
    x = T.tf_embed_rows(pack(T, w), torch.tensor([3, 64], dtype=torch.int32, device="cuda"), ws=ws)
    assert T.tf_workspace_status(ws) == T.TF_E_INVALID_ARG
    assert torch.count_nonzero(x[1]) == 0


def test_argmax_rows_matches_numpy_first_maximum(T):
    rng = np.random.default_rng(720)
    M, N = 8, 151936
    vals = rng.integers(-50, 50, size=(M, N)).astype(np.float32)  # many ties: the lowest index wins
    vals[2, :] = -1.0
    vals[2, 1234], vals[2, 99999] = 7.0, 7.0
    vals[3, :] = 0.0
    vals[3, 5] = -0.0  # -0 equals +0: index 0 wins
    v = dev_bf16(synth.f32_to_bf16_bits(vals))
    idx = T.tf_argmax_rows(v).cpu().numpy()
    np.testing.assert_array_equal(idx, np.argmax(vals, axis=1))
    assert idx[2] == 1234 and idx[3] == 0


def _decoder(T, cfg):
    layers = []
    for L in cfg["layers"]:
        layers.append({"qkv": pack(T, L["qkv"]), "o": pack(T, L["o"]), "gate": pack(T, L["gate"]),
                       "up": pack(T, L["up"]), "down": pack(T, L["down"]),
                       "attn_norm": dev_bf16(L["attn_norm"]), "mlp_norm": dev_bf16(L["mlp_norm"])})
    d = cfg["dims"]
    return T.Decoder(layers, dev_bf16(cfg["final_norm"]), pack(T, cfg["readout"]), d["d_model"], d["d_ff"],
                     d["q_dim"], d["kv_dim"], cfg["eps"])


def _check_generation(T, dec, n_new, seed):
    # a prompt that holds the continuation the model will produce: plain decoding from
    # a start token, then the prompt [start, first 3/4 of it, start]; generating from
    # that prompt repeats the continuation, so the drafts are mostly right
    rng = np.random.default_rng(seed)
    start = int(rng.integers(0, dec.readout.N))
    cont, steps0, acc0 = T.tf_generate_greedy(dec, [start], n_new, max_draft=0)
    assert len(cont) == n_new and steps0 == n_new and acc0 == 0
    # every token is the argmax of one decoder step on the previous token's embedding
    prev = [start] + cont[:-1]
    ids = torch.tensor(prev[:8], dtype=torch.int32, device="cuda")
    logits = T.tf_decode_step_run(dec, T.tf_embed_rows(dec.readout, ids))
    assert T.tf_argmax_rows(logits).cpu().tolist() == cont[:8]
    prompt = [start] + cont[: 3 * n_new // 4] + [start]
    plain, steps_p, _ = T.tf_generate_greedy(dec, prompt, n_new, max_draft=0)
    spec, steps_s, accepted = T.tf_generate_greedy(dec, prompt, n_new, max_draft=7)
    assert spec == plain  # the verify block does not change the text
    assert plain == cont  # a memoryless model: the prompt's tail token decides
    assert accepted > 0 and steps_s < steps_p and steps_s + accepted == n_new
    return steps_s, accepted


def test_greedy_generation_with_drafts_equals_plain_decoding_small(T):
    cfg = synth.decoder(seed=38, n_layers=2, d_model=256, d_ff=384, n_q_heads=4, n_kv_heads=2, head_dim=64,
                        vocab=1000, M=1)
    _check_generation(T, _decoder(T, cfg), 48, seed=1)


@pytest.mark.parametrize("chain", [1, 2])
def test_greedy_generation_with_drafts_equals_plain_decoding_full_size(T, chain):
    # 28 layers, model_dim 1024, hidden 3072, tied readout 151,936 x 1024; both step
    # implementations (one kernel per projection, the single persistent kernel)
    cfg = synth.decoder(M=1)
    T.tune_set(T.TF_TUNE_CHAIN, chain)
    try:
        _check_generation(T, _decoder(T, cfg), 24, seed=2)
    finally:
        T.tune_set(T.TF_TUNE_CHAIN, -1)


def test_generation_reuses_and_separates_its_step_graphs(T):
    # a step is replayed from a graph cached per (decoder, workspace, block length): the
    # same call twice on one workspace (replayed), a second decoder on that workspace
    # (its own graphs), the first again, and the first on another workspace give the
    # tokens of a fresh run each time
    cfg_a = synth.decoder(seed=61, n_layers=2, d_model=256, d_ff=384, n_q_heads=4, n_kv_heads=2, head_dim=64,
                          vocab=1000, M=1)
    cfg_b = synth.decoder(seed=62, n_layers=2, d_model=256, d_ff=384, n_q_heads=4, n_kv_heads=2, head_dim=64,
                          vocab=1000, M=1)
    dec_a, dec_b = _decoder(T, cfg_a), _decoder(T, cfg_b)
    ws = T.workspace(T.tf_generate_workspace_bytes(dec_a))
    prompt = [5, 17, 3, 5, 17]
    ref_a = T.tf_generate_greedy(dec_a, prompt, 20, max_draft=7, ws=ws)
    ref_b = T.tf_generate_greedy(dec_b, prompt, 20, max_draft=7, ws=T.workspace(T.tf_generate_workspace_bytes(dec_b)))
    assert ref_a[0] != ref_b[0]  # two different models
    assert T.tf_generate_greedy(dec_a, prompt, 20, max_draft=7, ws=ws) == ref_a
    assert T.tf_generate_greedy(dec_b, prompt, 20, max_draft=7, ws=ws) == ref_b
    assert T.tf_generate_greedy(dec_a, prompt, 20, max_draft=7, ws=ws) == ref_a
    ws2 = T.workspace(T.tf_generate_workspace_bytes(dec_a))
    assert T.tf_generate_greedy(dec_a, prompt, 20, max_draft=7, ws=ws2) == ref_a
    # plain decoding agrees token by token
    assert T.tf_generate_greedy(dec_a, prompt, 20, max_draft=0, ws=ws)[0] == ref_a[0]
