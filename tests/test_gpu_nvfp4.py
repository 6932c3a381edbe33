"""GPU parity of the NVFP4 weight code (E2M1 codes, an E4M3 scale per 16 columns, an
fp32 scale per matrix; TensorFold page, "qualified" model table: NVFP4 checkpoints)
against the fp64 oracle: packing, the exact value of every (code, scale) pair, and
the projections that accept it."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, dev_bf16, host_f64, tol_linear, tol_swiglu
from skinny_gemm_bit_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    from skinny_gemm_bit_gb300 import build
    build.build()
    from skinny_gemm_bit_gb300 import tfq
    return tfq


def pack4(T, w):
    return T.tf_qlinear_pack_nvfp4(w["codes"], w["scales"], float(w["gscale"]))


def x_bf16(rng, M, K):
    return synth.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))


# ------------------------------------------------------------------ packing

@pytest.mark.parametrize("N,K", [(3072, 1024), (1000, 640), (1, 64), (17, 192)])
def test_pack_roundtrip_bit_exact(T, N, K):
    w = synth.nvfp4_weights(np.random.default_rng(300 + N), N, K)
    qw = pack4(T, w)
    T.tf_qweight_check(qw)
    assert qw.code == T.TF_CODE_NVFP4 and qw.desc.group == 16 and qw.desc.global_scale == np.float32(w["gscale"])
    codes, scales, _ = T.tf_qlinear_unpack_debug(qw)
    assert np.array_equal(codes.cpu().numpy(), w["codes"]) and np.array_equal(scales.cpu().numpy(), w["scales"])


def test_stale_global_scale_is_refused(T):
    w = synth.nvfp4_weights(np.random.default_rng(5), 32, 128)
    qw = pack4(T, w)
    qw.desc.global_scale = 2.0
    with pytest.raises(T.TfqError) as e:
        T.tf_qweight_check(qw)
    assert e.value.status == T.TF_E_BAD_PACK


# ------------------------------------------------------------------ every value

@pytest.mark.parametrize("path", ["f16", "bf16"])
def test_every_code_and_scale_pair_is_exact(T, path):
    # row n has block-scale byte n everywhere (NaN for 0x7F and 0xFF, negative from
    # 0x80, subnormal for exponent 0) and code bytes (j + n) % 256, so the 256 rows see
    # all 65536 (code, scale) pairs; unit-vector activations read single weights, which
    # the fp32 output holds exactly. The bf16 path is forced by a 2^17 activation in
    # row 7 (the CTA then keeps bf16 for all rows); 2^17 w is exact too.
    N, K = 256, 512
    n = np.arange(N)[:, None]
    codes = ((np.arange(K // 2)[None, :] + n) % 256).astype(np.uint8)
    scales = np.repeat(np.arange(N, dtype=np.uint8)[:, None], K // 16, axis=1)
    w = {"code": "nvfp4", "codes": codes, "scales": scales, "gscale": np.float32(1.0), "N": N, "K": K}
    W = oracle.dequant(w)
    qw = pack4(T, w)
    big = 2.0 ** 17 if path == "bf16" else 1.0
    got = np.empty((N, K))
    for k0 in range(0, K, 8):
        xf = np.zeros((8, K), np.float32)
        for m in range(8):
            xf[m, k0 + m] = big if m == 7 else 1.0
        y = host_f64(T.tf_qlinear_run(qw, dev_bf16(synth.f32_to_bf16_bits(xf)), out_dtype=torch.float32))
        got[:, k0:k0 + 7] = y[:7].T
        got[:, k0 + 7] = y[7] / big
    np.testing.assert_array_equal(got, W)


# ------------------------------------------------------------------ random parity

SHAPES = [  # (M, K, N)
    (1, 1024, 3072),
    (8, 1024, 3072),
    (8, 12800, 2560),     # wide verify projection: K splits
    (1, 12800, 2560),
    (3, 640, 1000),       # ragged N
    (5, 64, 1),           # one row, one group
    (8, 1024, 151936),    # readout size
]


@pytest.mark.parametrize("M,K,N", SHAPES)
def test_qlinear_matches_oracle(T, M, K, N):
    rng = np.random.default_rng(M * 7919 + N)
    w = synth.nvfp4_weights(rng, N, K)
    x = x_bf16(rng, M, K)
    y = T.tf_qlinear_run(pack4(T, w), dev_bf16(x))
    y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(x), w)
    assert_close(host_f64(y), y_ref, tol_linear(ad), f"nvfp4 M={M} K={K} N={N}")


@pytest.mark.parametrize("M", [1, 8])
def test_rmsnorm_residual_fp32(T, M):
    rng = np.random.default_rng(310 + M)
    K, N = 1024, 2000
    w = synth.nvfp4_weights(rng, N, K)
    x = x_bf16(rng, M, K)
    g = synth.gamma(rng, K)
    res = x_bf16(rng, M, N)
    qw = pack4(T, w)
    xn = oracle.rmsnorm(oracle.bf16_to_f64(x), oracle.bf16_to_f64(g), 1e-6)
    y_ref, ad = oracle.qlinear(xn, w)
    y = T.tf_qlinear_run(qw, dev_bf16(x), gamma=dev_bf16(g), eps=1e-6, out_dtype=torch.float32)
    assert_close(host_f64(y), y_ref, tol_linear(ad), "norm fp32")
    yr = T.tf_qlinear_run(qw, dev_bf16(x), gamma=dev_bf16(g), eps=1e-6, residual=dev_bf16(res))
    ref_r = y_ref + oracle.bf16_to_f64(res)
    assert_close(host_f64(yr), ref_r, tol_linear(ad) + 2.0 ** -8 * np.abs(ref_r), "norm + residual")


@pytest.mark.parametrize("M,K,N,norm", [(8, 12800, 2560, False), (1, 1024, 3072, True), (3, 640, 1000, False)])
def test_rht_matches_oracle(T, M, K, N, norm):
    rng = np.random.default_rng(320 + M + N)
    w = synth.nvfp4_weights(rng, N, K)
    x = x_bf16(rng, M, K)
    signs = synth.rht_signs(rng, K)
    g = synth.gamma(rng, K) if norm else None
    xin = oracle.bf16_to_f64(x)
    if norm:
        xin = oracle.rmsnorm(xin, oracle.bf16_to_f64(g), 1e-6)
    y_ref, ad = oracle.qlinear(oracle.rht(xin, signs), w)
    y = T.tf_qlinear_run_rht(pack4(T, w), dev_bf16(x), torch.from_numpy(signs).cuda(),
                             gamma=dev_bf16(g) if norm else None, eps=1e-6, out_dtype=torch.float32)
    assert_close(host_f64(y), y_ref, tol_linear(ad), f"rht M={M} K={K} N={N}")


@pytest.mark.parametrize("M", [1, 8])
def test_fused_gateup_swiglu(T, M):
    rng = np.random.default_rng(330 + M)
    K, N = 1024, 3072
    gw, uw = synth.nvfp4_weights(rng, N, K), synth.nvfp4_weights(rng, N, K)
    uw["gscale"] = np.float32(0.0025)  # the two matrices carry different global scales
    x = x_bf16(rng, M, K)
    g = synth.gamma(rng, K)
    ref = oracle.gateup(oracle.bf16_to_f64(x), gw, uw, oracle.bf16_to_f64(g), 1e-6)
    h = T.tf_qmlp_gateup_run(pack4(T, gw), pack4(T, uw), dev_bf16(x), gamma=dev_bf16(g), eps=1e-6)
    assert_close(host_f64(h), ref["h"], tol_swiglu(ref["g"], ref["u"], ref["g_abs"], ref["u_abs"]), "gate/up")


@pytest.mark.parametrize("case", ["near_65536", "beyond_65536", "tiny"])
def test_activation_edges(T, case):
    # fp16 activations when every staged value converts exactly (|x| < 65536, finite),
    # else bf16; fp16 subnormals round
    rng = np.random.default_rng(["near_65536", "beyond_65536", "tiny"].index(case) + 340)
    M, K, N = 3, 1024, 4096
    xf = rng.standard_normal((M, K)).astype(np.float32)
    if case == "near_65536":
        xf[0, 5], xf[2, 700] = 65280.0, -61440.0
    elif case == "beyond_65536":
        xf[1, 17] = 131072.0
    else:
        xf *= 1e-6
    x = synth.f32_to_bf16_bits(xf)
    w = synth.nvfp4_weights(rng, N, K)
    y = T.tf_qlinear_run(pack4(T, w), dev_bf16(x), out_dtype=torch.float32)
    y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(x), w)
    assert_close(host_f64(y), y_ref, tol_linear(ad), case)


@pytest.mark.parametrize("warps,chunk", [(8, 8), (16, 4), (4, 16)])
def test_worker_shapes_match(T, warps, chunk):
    # workers a CTA and tiles a chunk as tuned (16 workers' ring slots do not fit at
    # K = 12800 with two staged K splits: the planner falls back to lock-step teams)
    rng = np.random.default_rng(350 + warps)
    M, K, N = 8, 12800, 2560
    w = synth.nvfp4_weights(rng, N, K)
    x = x_bf16(rng, M, K)
    qw = pack4(T, w)
    T.tune_set(T.TF_TUNE_WARPS, warps)
    T.tune_set(T.TF_TUNE_STAGE_GROUPS, chunk)
    try:
        y = T.tf_qlinear_run(qw, dev_bf16(x), out_dtype=torch.float32)
    finally:
        T.tune_set(T.TF_TUNE_WARPS, -1)
        T.tune_set(T.TF_TUNE_STAGE_GROUPS, -1)
    y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(x), w)
    assert_close(host_f64(y), y_ref, tol_linear(ad), f"warps {warps} chunk {chunk}")


def test_rows_are_independent_bit_exact(T):
    # a row's result does not depend on the other rows of the block (all finite, below 2^16)
    rng = np.random.default_rng(360)
    K, N = 1024, 151936
    w = synth.nvfp4_weights(rng, N, K)
    x = x_bf16(rng, 8, K)
    g = synth.gamma(rng, K)
    qw = pack4(T, w)
    y8 = T.tf_qlinear_run(qw, dev_bf16(x), gamma=dev_bf16(g), eps=1e-6)
    for m in (0, 5):
        y1 = T.tf_qlinear_run(qw, dev_bf16(x[m:m + 1]), gamma=dev_bf16(g), eps=1e-6)
        assert torch.equal(y1[0].view(torch.int16), y8[m].view(torch.int16)), m


@pytest.mark.parametrize("mode", [-1, 1, 2, 3, 4])
@pytest.mark.parametrize("M,K,N,dual", [(1, 1024, 3072, False), (8, 12800, 2560, False), (8, 1024, 3072, True),
                                        (3, 640, 1000, True)])
def test_every_schedule_matches(T, mode, M, K, N, dual):
    # the planner's choice, lock-step teams, warp workers, light teams with register-loaded
    # and with bulk-copied activations: NVFP4 tiles in the bf16 and fp16 tile math
    rng = np.random.default_rng(370 + M + N + mode)
    w = synth.nvfp4_weights(rng, N, K)
    x = x_bf16(rng, M, K)
    T.tune_set(T.TF_TUNE_MODE, mode)
    try:
        if dual:
            u = synth.nvfp4_weights(rng, N, K)
            g = synth.gamma(rng, K)
            h = T.tf_qmlp_gateup_run(pack4(T, w), pack4(T, u), dev_bf16(x), gamma=dev_bf16(g), eps=1e-6)
        else:
            y = T.tf_qlinear_run(pack4(T, w), dev_bf16(x), out_dtype=torch.float32)
    finally:
        T.tune_set(T.TF_TUNE_MODE, -1)
    if dual:
        ref = oracle.gateup(oracle.bf16_to_f64(x), w, u, oracle.bf16_to_f64(g), 1e-6)
        assert_close(host_f64(h), ref["h"], tol_swiglu(ref["g"], ref["u"], ref["g_abs"], ref["u_abs"]), f"mode {mode}")
    else:
        y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(x), w)
        assert_close(host_f64(y), y_ref, tol_linear(ad), f"mode {mode}")


# ------------------------------------------------------------------ decoder step and verify block

def test_embed_rows_nvfp4_bit_exact(T):
    # the token embedding from an NVFP4 tied readout: bf16 of the exact dequantised value
    rng = np.random.default_rng(380)
    N, K = 1000, 512
    w = synth.nvfp4_weights(rng, N, K)
    ids = np.array([0, 999, 17, 500, 999, 3], dtype=np.int32)
    ws = T.workspace(256)
    x = T.tf_embed_rows(pack4(T, w), torch.from_numpy(ids).cuda(), ws=ws)
    expect = synth.f32_to_bf16_bits(oracle.dequant(w)[ids].astype(np.float32))
    np.testing.assert_array_equal(x.cpu().view(torch.int16).numpy().view(np.uint16), expect)
    assert T.tf_workspace_status(ws) == T.TF_OK


@pytest.mark.parametrize("M", [1, 8])
def test_decoder_step_nvfp4_matches_oracle_stage_by_stage(T, M):
    # every stage of the step against the oracle applied to that stage's own inputs as
    # the GPU produced them (NVFP4 weights reach 6 * 448 * scale at the edge blocks, so
    # an earlier stage's rounding would otherwise dominate a later stage's bound); the
    # residual stages add 2^-8 |ref| for the bf16 rounding of the sum with the residual
    from test_gpu_verify import _decoder
    cfg = synth.decoder(seed=390 + M, n_layers=2, d_model=256, d_ff=384, n_q_heads=4, n_kv_heads=2, head_dim=64,
                        vocab=1000, M=M, code="nvfp4")
    dec = _decoder(T, cfg)
    d = cfg["dims"]
    QKV, D, F, q = d["q_dim"] + 2 * d["kv_dim"], d["d_model"], d["d_ff"], d["q_dim"]
    dbg = torch.zeros(T.tf_decode_step_debug_elems(dec, M), dtype=torch.bfloat16, device="cuda")
    logits = host_f64(T.tf_decode_step_run(dec, dev_bf16(cfg["x"]), debug=dbg))
    dbg_h = host_f64(dbg)
    per = M * (QKV + D + F + D)
    h = oracle.bf16_to_f64(cfg["x"])
    rel = 2.0 ** -8
    for l, L in enumerate(cfg["layers"]):
        blk = dbg_h[l * per:(l + 1) * per]
        qkv = blk[:M * QKV].reshape(M, QKV)
        h1 = blk[M * QKV:M * (QKV + D)].reshape(M, D)
        a = blk[M * (QKV + D):M * (QKV + D + F)].reshape(M, F)
        h2 = blk[M * (QKV + D + F):].reshape(M, D)
        # a plain projection's bf16 output (2^-9 |y| <= 2^-9 sum |x w|) is inside the projection bound itself
        ref, ad = oracle.qlinear(oracle.rmsnorm(h, oracle.bf16_to_f64(L["attn_norm"]), cfg["eps"]), L["qkv"])
        assert_close(qkv, ref, tol_linear(ad), f"layer {l} qkv")
        o, ad = oracle.qlinear(qkv[:, :q], L["o"])
        assert_close(h1, h + o, tol_linear(ad) + rel * np.abs(h + o), f"layer {l} h1")
        gu = oracle.gateup(h1, L["gate"], L["up"], oracle.bf16_to_f64(L["mlp_norm"]), cfg["eps"])
        assert_close(a, gu["h"], tol_swiglu(gu["g"], gu["u"], gu["g_abs"], gu["u_abs"]), f"layer {l} swiglu")
        dn, ad = oracle.qlinear(a, L["down"])
        assert_close(h2, h1 + dn, tol_linear(ad) + rel * np.abs(h1 + dn), f"layer {l} h2")
        h = h2
    ref, ad = oracle.qlinear(oracle.rmsnorm(h, oracle.bf16_to_f64(cfg["final_norm"]), cfg["eps"]), cfg["readout"])
    assert_close(logits, ref, tol_linear(ad), "logits")


def test_generation_with_drafts_nvfp4_equals_plain_decoding(T):
    from test_gpu_verify import _check_generation, _decoder
    cfg = synth.decoder(seed=395, n_layers=2, d_model=256, d_ff=384, n_q_heads=4, n_kv_heads=2, head_dim=64,
                        vocab=1000, M=1, code="nvfp4")
    _check_generation(T, _decoder(T, cfg), 48, seed=3)


def test_chained_step_refuses_nvfp4(T):
    # the single-kernel step reads affine codes only: asked for, it is refused by name
    cfg = synth.decoder(seed=396, n_layers=1, d_model=256, d_ff=384, n_q_heads=4, n_kv_heads=2, head_dim=64,
                        vocab=1000, M=1, code="nvfp4")
    from test_gpu_verify import _decoder
    dec = _decoder(T, cfg)
    T.tune_set(T.TF_TUNE_CHAIN, 2)
    try:
        with pytest.raises(T.TfqError) as e:
            T.tf_decode_step_run(dec, dev_bf16(cfg["x"]))
        assert e.value.status == T.TF_E_UNSUPPORTED_SHAPE
    finally:
        T.tune_set(T.TF_TUNE_CHAIN, -1)


# ------------------------------------------------------------------ MoE experts

def test_pack_experts_roundtrip(T):
    # a stack of 5 expert matrices with their own fp32 scales: codes, block scales and the
    # scale table come back bit for bit
    w = synth.nvfp4_weights(np.random.default_rng(501), 40, 128, batch=5)
    qw = T.tf_qlinear_pack_nvfp4(w["codes"], w["scales"], w["gscale"])
    T.tf_qweight_check(qw)
    assert qw.batch == 5 and qw.code == T.TF_CODE_NVFP4
    codes, scales, gs = T.tf_qlinear_unpack_debug(qw)
    assert np.array_equal(codes.cpu().numpy(), w["codes"]) and np.array_equal(scales.cpu().numpy(), w["scales"])
    assert np.array_equal(gs.cpu().numpy(), w["gscale"])
    assert len(set(w["gscale"].tolist())) > 1  # the experts' scales differ, so pairing them matters


def _check_moe_nvfp4(T, cfg):
    from test_gpu_moe_decode import _check_moe
    _check_moe(T, cfg)


def test_moe_nvfp4_full_size(T):
    # M=8 rows, 128 NVFP4 experts, top-8, hidden 2048, expert intermediate 768
    _check_moe_nvfp4(T, synth.moe_layer(code="nvfp4"))


@pytest.mark.parametrize("M,E,top_k", [(1, 128, 8), (3, 16, 4), (8, 8, 8), (2, 5, 1)])
def test_moe_nvfp4_small(T, M, E, top_k):
    _check_moe_nvfp4(T, synth.moe_layer(seed=60 + M + E, M=M, E=E, top_k=top_k, hidden=256, inter=128, code="nvfp4"))
