"""GPU parity of the MoE layer and the chained decoder-step weight stream."""
import numpy as np
import pytest
import torch

import oracle
from parity import (BF16_REL, assert_close, dev_bf16, dev_f32, host_f64, moe_tolerance, pack, tol_linear,
                    tol_swiglu)
from skinny_gemm_bit_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    from skinny_gemm_bit_gb300 import build
    build.build()
    from skinny_gemm_bit_gb300 import tfq
    return tfq


# ------------------------------------------------------------------ MoE

def _run_moe(T, cfg, ws=None):
    gate, up, down = pack(T, cfg["gate"]), pack(T, cfg["up"]), pack(T, cfg["down"])
    y, idx, w = T.tf_qmoe_run(gate, up, down, dev_f32(cfg["logits"]), dev_bf16(cfg["x"]), cfg["top_k"], ws=ws)
    return y, idx, w


def _check_moe(T, cfg):
    y, idx, w = _run_moe(T, cfg)
    ref = oracle.moe(oracle.bf16_to_f64(cfg["x"]), cfg["logits"], cfg["gate"], cfg["up"], cfg["down"],
                     cfg["top_k"])
    idx = idx.cpu().numpy()
    w = w.cpu().numpy().astype(np.float64)
    assert np.array_equal(idx, ref["idx"])
    np.testing.assert_allclose(w, ref["w"], rtol=1e-6, atol=0)
    assert_close(host_f64(y), ref["y"], moe_tolerance(ref, cfg["down"], w), "moe y")


@pytest.mark.parametrize("bits", [4, 8])
def test_moe_full_size(T, bits):
    # M=8 rows, 128 experts, top-8, hidden 2048, expert intermediate 768
    _check_moe(T, synth.moe_layer(bits=bits))


@pytest.mark.parametrize("M,E,top_k", [(1, 128, 8), (3, 16, 4), (8, 8, 8), (2, 5, 1)])
def test_moe_small(T, M, E, top_k):
    _check_moe(T, synth.moe_layer(seed=40 + M + E, M=M, E=E, top_k=top_k, hidden=256, inter=128))


def test_moe_with_ties_routes_to_lower_index(T):
    cfg = synth.moe_layer(seed=44, M=4, E=32, top_k=4, hidden=128, inter=64)
    cfg["logits"] = np.random.default_rng(3).integers(-2, 3, size=(4, 32)).astype(np.float32)
    _check_moe(T, cfg)


def test_moe_repeat_is_byte_identical(T):
    cfg = synth.moe_layer(seed=45)
    gate, up, down = pack(T, cfg["gate"]), pack(T, cfg["up"]), pack(T, cfg["down"])
    lg, x = dev_f32(cfg["logits"]), dev_bf16(cfg["x"])
    ws = T.workspace(T.tf_qmoe_workspace_bytes(gate, up, down, 8, 8))
    outs = [T.tf_qmoe_run(gate, up, down, lg, x, 8, ws=ws)[0].clone() for _ in range(5)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert T.tf_workspace_status(ws) == T.TF_OK


def test_moe_expert_down_projection_exact(T):
    # The expert projections of the MoE layer (gathered rows, per-slot problems) with
    # every product and sum exact: x = 1, bias-only gate and up (scale 0) with
    # g = 2048 / 16 = 128 and u = 2048 / 1024 = 2, so h = silu(128) * 2 = 256 exactly (the
    # exponential underflows in fp32 and fp64 alike) and the bf16 h is exact; random 4-bit
    # down codes with scale 1 and integer biases give integer sums far below 2^24; top-1
    # routing weighs each row's expert by exactly 1. The output is then the oracle's
    # integer rounded once to bf16, bit for bit.
    rng = np.random.default_rng(47)
    M, E, H, I = 8, 16, 2048, 768
    cfg = synth.moe_layer(seed=46, M=M, E=E, top_k=1, hidden=H, inter=I)
    cfg["x"] = synth.f32_to_bf16_bits(np.ones((M, H), np.float32))
    for name, beta in (("gate", 1 / 16), ("up", 1 / 1024)):
        cfg[name]["scales"][:] = 0
        cfg[name]["biases"][:] = synth.f32_to_bf16_bits(np.float32(beta))
    dn = cfg["down"]
    dn["scales"][:] = 0x3F80
    dn["biases"] = synth.f32_to_bf16_bits(rng.integers(-12, -3, size=dn["scales"].shape).astype(np.float32))
    y, idx, w = _run_moe(T, cfg)
    ref = oracle.moe(oracle.bf16_to_f64(cfg["x"]), cfg["logits"], cfg["gate"], cfg["up"], cfg["down"], 1)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.all(w.cpu().numpy() == 1.0)
    assert all(s["h"].min() == 256.0 and s["h"].max() == 256.0 for row in ref["slots"] for s in row)
    assert np.abs(ref["y"]).max() < 2 ** 24 and np.all(ref["y"] == np.round(ref["y"]))
    expect = synth.f32_to_bf16_bits(ref["y"].astype(np.float32))
    got = y.cpu().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, expect)


# ------------------------------------------------------------------ decoder step

def _pack_decoder(T, cfg):
    layers = []
    for L in cfg["layers"]:
        layers.append({"qkv": pack(T, L["qkv"]), "o": pack(T, L["o"]), "gate": pack(T, L["gate"]),
                       "up": pack(T, L["up"]), "down": pack(T, L["down"]),
                       "attn_norm": dev_bf16(L["attn_norm"]), "mlp_norm": dev_bf16(L["mlp_norm"])})
    d = cfg["dims"]
    return T.Decoder(layers, dev_bf16(cfg["final_norm"]), pack(T, cfg["readout"]), d["d_model"], d["d_ff"],
                     d["q_dim"], d["kv_dim"], cfg["eps"])


def _oracle_layers(cfg):
    return [{k: (oracle.bf16_to_f64(v) if k.endswith("norm") else v) for k, v in L.items()} for L in cfg["layers"]]


def _check_decoder(T, cfg, M, readout_rows=None):
    dec = _pack_decoder(T, cfg)
    d = cfg["dims"]
    x = dev_bf16(cfg["x"])
    dbg = torch.zeros(T.tf_decode_step_debug_elems(dec, M), dtype=torch.bfloat16, device="cuda")
    logits = T.tf_decode_step_run(dec, x, debug=dbg)
    logits_nodbg = T.tf_decode_step_run(dec, x)
    assert torch.equal(logits, logits_nodbg)
    ref = oracle.decode_step(oracle.bf16_to_f64(cfg["x"]), _oracle_layers(cfg),
                             oracle.bf16_to_f64(cfg["final_norm"]), cfg["readout"], d["q_dim"], cfg["eps"],
                             readout_rows=readout_rows)
    QKV = d["q_dim"] + 2 * d["kv_dim"]
    D, F = d["d_model"], d["d_ff"]
    per = M * (QKV + D + F + D)
    dbg_h = host_f64(dbg)
    tol_h = np.zeros((M, D))  # bound of the residual stream entering the layer
    for l, st in enumerate(ref["stages"]):
        blk = dbg_h[l * per:(l + 1) * per]
        qkv = blk[:M * QKV].reshape(M, QKV)
        h1 = blk[M * QKV:M * (QKV + D)].reshape(M, D)
        a = blk[M * (QKV + D):M * (QKV + D + F)].reshape(M, F)
        h2 = blk[M * (QKV + D + F):].reshape(M, D)
        assert_close(qkv, st["qkv"], tol_linear(st["qkv_abs"]), f"layer {l} qkv")
        tol_h1 = tol_h + tol_linear(st["o_abs"]) + BF16_REL * np.abs(st["h1"])
        assert_close(h1, st["h1"], tol_h1, f"layer {l} h1")
        gu = st["gu"]
        assert_close(a, gu["h"], tol_swiglu(gu["g"], gu["u"], gu["g_abs"], gu["u_abs"]), f"layer {l} swiglu")
        tol_h = tol_h1 + tol_linear(st["d_abs"]) + BF16_REL * np.abs(st["h2"])
        assert_close(h2, st["h2"], tol_h, f"layer {l} h2")
    lg = host_f64(logits)
    if readout_rows is not None:
        lg = lg[:, readout_rows]
    assert_close(lg, ref["logits"], tol_linear(ref["logits_abs"]), "logits")


@pytest.mark.parametrize("per_projection", [False, True])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_decoder_small(T, M, per_projection):
    # the whole step in one persistent kernel (required, so no silent fallback), or one
    # kernel per projection
    cfg = synth.decoder(seed=30 + M, n_layers=3, d_model=256, d_ff=384, n_q_heads=4, n_kv_heads=2, head_dim=64,
                        vocab=1000, M=M)
    T.tune_set(T.TF_TUNE_CHAIN, 1 if per_projection else 2)
    try:
        _check_decoder(T, cfg, M)
    finally:
        T.tune_set(T.TF_TUNE_CHAIN, -1)


@pytest.mark.parametrize("per_projection", [False, True])
def test_decoder_step_rows_are_independent_bit_exact(T, per_projection):
    # a row's logits are the same bits whether it runs alone or in a block of 8 (the
    # property a greedy verify block needs: its predictions equal one-row decoding)
    cfg = synth.decoder(seed=37, n_layers=2, d_model=1024, d_ff=1024, n_q_heads=4, n_kv_heads=2, head_dim=128,
                        vocab=4096, M=8)
    dec = _pack_decoder(T, cfg)
    x = dev_bf16(cfg["x"])
    T.tune_set(T.TF_TUNE_CHAIN, 1 if per_projection else 2)
    try:
        y8 = T.tf_decode_step_run(dec, x)
        for m in range(8):
            y1 = T.tf_decode_step_run(dec, x[m:m + 1])
            assert torch.equal(y1[0], y8[m]), m
    finally:
        T.tune_set(T.TF_TUNE_CHAIN, -1)


def test_decoder_step_leaves_workspace_clean_and_repeats_exactly(T):
    cfg = synth.decoder(seed=39, n_layers=2, d_model=256, d_ff=384, n_q_heads=4, n_kv_heads=2, head_dim=64,
                        vocab=1000, M=4)
    dec = _pack_decoder(T, cfg)
    x = dev_bf16(cfg["x"])
    ws = T.workspace(T.tf_decode_step_workspace_bytes(dec, 4))
    outs = [T.tf_decode_step_run(dec, x, ws=ws).clone() for _ in range(3)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert T.tf_workspace_status(ws) == T.TF_OK


@pytest.mark.parametrize("chain", [-1, 2])
@pytest.mark.parametrize("M", [1, 8])
def test_decoder_full_size(T, M, chain):
    # 28 layers, model_dim 1024, hidden 3072, 16 q / 8 kv heads of 128, tied readout 151,936 x 1024,
    # through the default chain of per-projection kernels (chain -1: what the benchmark times)
    # and through the single-kernel step (chain 2, required)
    cfg = synth.decoder(M=M)
    rows = np.sort(np.random.default_rng(9).choice(151936, size=512, replace=False))
    rows = np.concatenate([rows, [0, 151935]])
    T.tune_set(T.TF_TUNE_CHAIN, chain)
    try:
        _check_decoder(T, cfg, M, readout_rows=np.unique(rows))
    finally:
        T.tune_set(T.TF_TUNE_CHAIN, -1)
