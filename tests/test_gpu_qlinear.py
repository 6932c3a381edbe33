"""GPU parity of packing and the single / fused projections against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity import (ATOL, BF16_REL, EPS, assert_close, dev_bf16, host_f64, pack, tol_linear, tol_swiglu)
from skinny_gemm_bit_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    from skinny_gemm_bit_gb300 import build
    build.build()
    from skinny_gemm_bit_gb300 import tfq
    return tfq


def _w_host(T, qw):
    wq, s, b = T.tf_qlinear_unpack_debug(qw)
    torch.cuda.synchronize()
    return (wq.cpu().numpy().view(np.uint32), s.cpu().numpy().view(np.uint16), b.cpu().numpy().view(np.uint16))


# ------------------------------------------------------------------ packing

@pytest.mark.parametrize("bits,N,K,batch", [(4, 3072, 1024, 1), (4, 1000, 640, 1), (8, 200, 192, 1),
                                            (4, 48, 128, 5), (8, 17, 64, 3), (4, 1, 64, 1)])
def test_pack_roundtrip_bit_exact(T, bits, N, K, batch):
    rng = np.random.default_rng(100 + N)
    w = synth.quant_weights(rng, N, K, bits, batch=None if batch == 1 else batch)
    qw = pack(T, w)
    T.tf_qweight_check(qw)
    wq, s, b = _w_host(T, qw)
    assert np.array_equal(wq, w["wq"]) and np.array_equal(s, w["scales"]) and np.array_equal(b, w["biases"])


def test_pack_roundtrip_every_32bit_word(T):
    # all 2^32 word values through pack -> unpack, in chunks, 4-bit and 8-bit
    K = 1024
    chunk = 1 << 27
    for bits in (4, 8):
        words_per_row = K * bits // 32
        rows = chunk // words_per_row
        s = torch.zeros((rows, K // 64), dtype=torch.int16, device="cuda")
        for c in range((1 << 32) // chunk):
            wq = (torch.arange(chunk, dtype=torch.int64, device="cuda") + c * chunk).to(torch.int32)
            wq = wq.view(rows, words_per_row)
            qw = T.tf_qlinear_pack(wq, s, s, bits)
            back, _, _ = T.tf_qlinear_unpack_debug(qw)
            assert torch.equal(back, wq), f"bits={bits} chunk {c}"
            del qw, back, wq
    torch.cuda.synchronize()


def test_stale_descriptor_is_refused(T):
    w = synth.quant_weights(np.random.default_rng(1), 64, 128, 4)
    qw = pack(T, w)
    qw.desc.N = 80
    qw.desc.n_pad = 80
    qw.desc.matrix_bytes = 5 * 2 * 576
    with pytest.raises(T.TfqError) as e:
        T.tf_qweight_check(qw)
    assert e.value.status == T.TF_E_BAD_PACK


# ------------------------------------------------------------------ exact cases

def test_hand_case_exact(T):
    M, K, N = 4, 64, 8
    q = np.array([[(n + k) % 16 for k in range(K)] for n in range(N)])
    s = synth.f32_to_bf16_bits(np.array([2.0 ** -n for n in range(N)], np.float32))[:, None]
    b = synth.f32_to_bf16_bits(np.array([-n / 8 for n in range(N)], np.float32))[:, None]
    w = {"wq": synth.pack_codes(q, 4), "scales": s, "biases": b, "N": N, "K": K, "bits": 4}
    x = synth.f32_to_bf16_bits(np.array([[m + 1] * K for m in range(M)], np.float32))
    y = T.tf_qlinear_run(pack(T, w), dev_bf16(x), out_dtype=torch.float32)
    expect = np.array([[(m + 1) * (480 * 2.0 ** -n - 8 * n) for n in range(N)] for m in range(M)])
    assert np.array_equal(host_f64(y), expect)


def _bf16_accumulating_dot(x, w):
    acc = np.float32(0)
    for a, c in zip(x, w):
        v = np.array([acc + np.float32(a) * np.float32(c)], dtype=np.float32)
        acc = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(v))[0]
    return float(acc)


@pytest.mark.parametrize("bits", [4, 8])
def test_fp32_exact_sum_gate(T, bits):
    # integer activations in [-256, 256], s = 1, integer b: every partial sum is an
    # integer below 2^24, so an fp32 accumulation is exact whatever its order.
    rng = np.random.default_rng(7 + bits)
    M, K, N = 8, 1024, 96
    xi = rng.integers(-256, 257, size=(M, K)).astype(np.float32)
    w = synth.quant_weights(rng, N, K, bits)
    w["scales"][:] = 0x3F80
    off = -8 if bits == 4 else -128
    w["biases"] = synth.f32_to_bf16_bits(rng.integers(off - 4, off + 5, size=w["scales"].shape).astype(np.float32))
    y_ref, _ = oracle.qlinear(xi.astype(np.float64), w)
    assert np.abs(y_ref).max() < 2 ** 24
    y = T.tf_qlinear_run(pack(T, w), dev_bf16(synth.f32_to_bf16_bits(xi)), out_dtype=torch.float32)
    assert np.array_equal(host_f64(y), y_ref)
    # planted control: a bf16-accumulating dot product does not meet this gate
    wd = oracle.dequant(w)
    assert any(_bf16_accumulating_dot(xi[0], wd[n]) != y_ref[0, n] for n in range(8))


def _exact_case(rng, M, K, N, bits, xmax):
    xi = rng.integers(-xmax, xmax + 1, size=(M, K)).astype(np.float32)
    w = synth.quant_weights(rng, N, K, bits)
    w["scales"][:] = 0x3F80
    off = -8 if bits == 4 else -128
    w["biases"] = synth.f32_to_bf16_bits(rng.integers(off - 4, off + 5, size=w["scales"].shape).astype(np.float32))
    return xi, w


# Every schedule the planner has (1: lock-step teams, 2: warp workers, 3: light teams,
# 4: light teams with bulk-copied rows, 5: streaming CTAs) on one unsplit and one
# split-K shape. |x| <= 128 (4-bit) / 64 (8-bit) keeps every partial sum of the warp
# workers' fp16 form (1024 + q and 1024 + 16 q code units) below 2^24, so the fp32
# sums are exact in every schedule and must equal the oracle.
@pytest.mark.parametrize("mode", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N", [(8, 1024, 96), (8, 12800, 256), (3, 4096, 1000)])
def test_fp32_exact_sum_gate_every_schedule(T, mode, bits, M, K, N):
    rng = np.random.default_rng(mode * 100 + bits * 10 + M + K)
    xi, w = _exact_case(rng, M, K, N, bits, 128 if bits == 4 else 64)
    y_ref, _ = oracle.qlinear(xi.astype(np.float64), w)
    assert np.abs(y_ref).max() < 2 ** 24
    T.tune_set(T.TF_TUNE_MODE, mode)
    try:
        y = T.tf_qlinear_run(pack(T, w), dev_bf16(synth.f32_to_bf16_bits(xi)), out_dtype=torch.float32)
    finally:
        T.tune_set(T.TF_TUNE_MODE, -1)
    assert np.array_equal(host_f64(y), y_ref), f"mode {mode}"


# NVFP4: integer x, every block scale byte 0x38 (E4M3 1.0) and a global scale of 1, so
# every weight is an E2M1 value (a multiple of 0.5 up to 6) and every partial sum a
# multiple of 0.5 far below 2^23: exact in fp32 on every schedule the code runs on.
@pytest.mark.parametrize("mode", [1, 2, 3, 4])
@pytest.mark.parametrize("M,K,N", [(8, 1024, 96), (8, 12800, 256)])
def test_nvfp4_exact_sum_gate(T, mode, M, K, N):
    rng = np.random.default_rng(900 + mode + K)
    xi = rng.integers(-256, 257, size=(M, K)).astype(np.float32)
    w = synth.nvfp4_weights(rng, N, K)
    w["scales"][:] = 0x38
    w["gscale"] = np.float32(1.0)
    y_ref, _ = oracle.qlinear(xi.astype(np.float64), w)
    assert np.all(y_ref * 2 == np.round(y_ref * 2)) and np.abs(y_ref).max() < 2 ** 22
    T.tune_set(T.TF_TUNE_MODE, mode)
    try:
        qw = T.tf_qlinear_pack_nvfp4(w["codes"], w["scales"], float(w["gscale"]))
        y = T.tf_qlinear_run(qw, dev_bf16(synth.f32_to_bf16_bits(xi)), out_dtype=torch.float32)
    finally:
        T.tune_set(T.TF_TUNE_MODE, -1)
    assert np.array_equal(host_f64(y), y_ref), f"mode {mode}"


# ------------------------------------------------------------------ random parity

SHAPES = [  # (M, K, N, bits)
    (1, 1024, 3072, 4),      # single 4-bit projection, decode
    (8, 1024, 3072, 4),
    (8, 12800, 2560, 4),     # wide verify projection
    (1, 12800, 2560, 4),
    (3, 640, 1000, 4),       # ragged N, several tiles
    (5, 64, 1, 4),           # one row, one group
    (8, 2048, 1024, 8),
    (2, 320, 333, 8),
]


@pytest.mark.parametrize("M,K,N,bits", SHAPES)
def test_qlinear_matches_oracle(T, M, K, N, bits):
    cfg = synth.single_projection(seed=M * 1000 + N, M=M, K=K, N=N, bits=bits)
    y = T.tf_qlinear_run(pack(T, cfg["w"]), dev_bf16(cfg["x"]))
    y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(cfg["x"]), cfg["w"])
    assert_close(host_f64(y), y_ref, tol_linear(ad), f"qlinear M={M} K={K} N={N} bits={bits}")


@pytest.mark.parametrize("M", [1, 4, 8])
def test_qlinear_rmsnorm_prologue(T, M):
    rng = np.random.default_rng(50 + M)
    K, N = 1024, 768
    x = synth.activations(rng, M, K)
    g = synth.gamma(rng, K)
    w = synth.quant_weights(rng, N, K, 4)
    y = T.tf_qlinear_run(pack(T, w), dev_bf16(x), gamma=dev_bf16(g), eps=1e-6)
    xn = oracle.rmsnorm(oracle.bf16_to_f64(x), oracle.bf16_to_f64(g), 1e-6)
    y_ref, ad = oracle.qlinear(xn, w)
    assert_close(host_f64(y), y_ref, tol_linear(ad), "rmsnorm + qlinear")


def test_qlinear_residual_and_strided_input(T):
    rng = np.random.default_rng(61)
    M, K, N = 6, 2048, 1024
    xfull = synth.activations(rng, M, K + 256)           # x is the first K columns (row stride K+256)
    res = synth.activations(rng, M, N)
    w = synth.quant_weights(rng, N, K, 4)
    xd = dev_bf16(xfull)[:, :K]
    y = T.tf_qlinear_run(pack(T, w), xd, residual=dev_bf16(res))
    y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(xfull)[:, :K], w)
    y_ref = y_ref + oracle.bf16_to_f64(res)
    assert_close(host_f64(y), y_ref, tol_linear(ad) + BF16_REL * np.abs(y_ref), "residual")


@pytest.mark.parametrize("M", [1, 8])
def test_fused_gateup_swiglu(T, M):
    cfg = synth.fused_gateup(M=M)
    h = T.tf_qmlp_gateup_run(pack(T, cfg["gate"]), pack(T, cfg["up"]), dev_bf16(cfg["x"]),
                             gamma=dev_bf16(cfg["gamma"]), eps=cfg["eps"])
    ref = oracle.gateup(oracle.bf16_to_f64(cfg["x"]), cfg["gate"], cfg["up"],
                        oracle.bf16_to_f64(cfg["gamma"]), cfg["eps"])
    tol = tol_swiglu(ref["g"], ref["u"], ref["g_abs"], ref["u_abs"])
    assert_close(host_f64(h), ref["h"], tol, f"gate/up M={M}")


def test_gateup_pre_activations_via_qlinear(T):
    # the same weights through the plain projection give gate and up themselves
    cfg = synth.fused_gateup(M=8)
    gamma = dev_bf16(cfg["gamma"])
    ref = oracle.gateup(oracle.bf16_to_f64(cfg["x"]), cfg["gate"], cfg["up"],
                        oracle.bf16_to_f64(cfg["gamma"]), cfg["eps"])
    for name, key in (("gate", "g"), ("up", "u")):
        y = T.tf_qlinear_run(pack(T, cfg[name]), dev_bf16(cfg["x"]), gamma=gamma, eps=cfg["eps"],
                             out_dtype=torch.float32)
        assert_close(host_f64(y), ref[key], tol_linear(ref[key + "_abs"]), name)


def test_gateup_ragged(T):
    rng = np.random.default_rng(71)
    M, K, N = 3, 320, 200
    x = synth.activations(rng, M, K)
    g = synth.quant_weights(rng, N, K, 4)
    u = synth.quant_weights(rng, N, K, 4)
    h = T.tf_qmlp_gateup_run(pack(T, g), pack(T, u), dev_bf16(x))
    ref = oracle.gateup(oracle.bf16_to_f64(x), g, u)
    assert_close(host_f64(h), ref["h"], tol_swiglu(ref["g"], ref["u"], ref["g_abs"], ref["u_abs"]), "ragged gate/up")


# ------------------------------------------------------------------ properties

def test_rows_are_independent_bit_exact(T):
    cfg = synth.wide_verify(M=8)
    qw = pack(T, cfg["w"])
    x = dev_bf16(cfg["x"])
    y8 = T.tf_qlinear_run(qw, x)
    for m in range(8):
        y1 = T.tf_qlinear_run(qw, x[m:m + 1])
        assert torch.equal(y1[0], y8[m]), m


def test_repeat_runs_are_byte_identical(T):
    cfg = synth.wide_verify(M=8)
    qw = pack(T, cfg["w"])
    x = dev_bf16(cfg["x"])
    ws = T.workspace(T.tf_qlinear_workspace_bytes(qw, 8))
    outs = [T.tf_qlinear_run(qw, x, ws=ws, out_dtype=torch.float32) for _ in range(5)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))
    assert T.tf_workspace_status(ws) == T.TF_OK


def test_guard_bytes_untouched(T):
    rng = np.random.default_rng(81)
    M, K, N = 8, 1024, 1000
    x = synth.activations(rng, M, K)
    w = synth.quant_weights(rng, N, K, 4)
    guard = 4096
    buf = torch.full((M * N + 2 * guard,), -12345.0, dtype=torch.float32, device="cuda")
    out = buf[guard:guard + M * N].view(M, N)
    T.tf_qlinear_run(pack(T, w), dev_bf16(x), out=out)
    assert torch.all(buf[:guard] == -12345.0) and torch.all(buf[guard + M * N:] == -12345.0)
    y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(x), w)
    assert_close(host_f64(out), y_ref, tol_linear(ad), "guarded output")


def test_nan_row_stays_in_its_row(T):
    rng = np.random.default_rng(91)
    M, K, N = 4, 1024, 512
    x = synth.activations(rng, M, K)
    x[2, 17] = 0x7FC0  # NaN
    w = synth.quant_weights(rng, N, K, 4)
    y = host_f64(T.tf_qlinear_run(pack(T, w), dev_bf16(x)))
    assert np.all(np.isnan(y[2]))
    assert np.all(np.isfinite(np.delete(y, 2, axis=0)))


def test_pdl_flag_gives_same_result(T):
    cfg = synth.single_projection(seed=5, M=8)
    qw = pack(T, cfg["w"])
    x = dev_bf16(cfg["x"])
    a = T.tf_qlinear_run(qw, x)
    torch.cuda._sleep(1000)  # an unrelated kernel right before
    b = T.tf_qlinear_run(qw, x, flags=T.TF_RUN_PDL)
    assert torch.equal(a, b)


def test_wait_timeout_is_reported_not_hung(T):
    ws = T.workspace(256)
    T.tf_selftest_wait_timeout(ws, 1_000_000)  # 1 ms bound on a barrier nothing arrives on
    assert T.tf_workspace_status(ws) == T.TF_E_TIMEOUT
    assert T.tf_workspace_status(ws) == T.TF_OK  # read clears it
    # the context is still usable
    cfg = synth.single_projection(seed=6, M=1, K=128, N=64)
    y = T.tf_qlinear_run(pack(T, cfg["w"]), dev_bf16(cfg["x"]))
    y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(cfg["x"]), cfg["w"])
    assert_close(host_f64(y), y_ref, tol_linear(ad), "after timeout")


@pytest.mark.parametrize("R,S", [(1, 1), (2, 5), (4, 2), (8, 4), (16, 10), (16, 1)])
def test_every_cta_shape_matches(T, R, S):
    # R row blocks side by side per round, S K-splits (S divides K/64 = 20)
    cfg = synth.single_projection(seed=R * 10 + S, M=8, K=1280, N=520)
    qw = pack(T, cfg["w"])
    T.tune_set(T.TF_TUNE_ROWBLOCKS, R)
    T.tune_set(T.TF_TUNE_SPLITK, S)
    try:
        y = T.tf_qlinear_run(qw, dev_bf16(cfg["x"]))
    finally:
        T.tune_set(T.TF_TUNE_ROWBLOCKS, -1)
        T.tune_set(T.TF_TUNE_SPLITK, -1)
    y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(cfg["x"]), cfg["w"])
    assert_close(host_f64(y), y_ref, tol_linear(ad), f"R={R} S={S}")


def test_shared_workspace_across_shapes_is_left_clean(T):
    # one workspace reused by projections of different shapes (as in a decoder
    # step): results equal those with a fresh workspace, and every call leaves
    # the workspace all-zero again (counters and partial slots)
    rng = np.random.default_rng(97)
    shapes = [(1024, 2048, 1), (4096, 1024, 1), (2560, 12800, 8), (1024, 3072, 3), (151936 // 8, 1024, 1),
              (777, 640, 5)]
    cases = []
    for N, K, M in shapes:
        w = pack(T, synth.quant_weights(rng, N, K, 4))
        x = dev_bf16(synth.activations(rng, M, K))
        cases.append((w, x, T.tf_qlinear_run(w, x, out_dtype=torch.float32)))
    ws = T.workspace(max(T.tf_qlinear_workspace_bytes(w, 8) for w, _, _ in cases))
    for _ in range(2):
        for w, x, ref in cases:
            y = T.tf_qlinear_run(w, x, ws=ws, out_dtype=torch.float32)
            assert torch.equal(y, ref)
            torch.cuda.synchronize()
            assert int(ws.count_nonzero()) == 0


@pytest.mark.parametrize("mode", [1, 2, 3, 4])
@pytest.mark.parametrize("M,K,N,bits,dual", [(8, 12800, 2560, 4, False), (1, 1024, 18992, 4, False),
                                              (3, 2048, 4096, 8, False), (8, 1024, 3072, 4, True),
                                              (2, 640, 6000, 4, True)])
def test_both_schedules_match(T, mode, M, K, N, bits, dual):
    # mode 1: lock-step teams; mode 2: warp workers with private ring slots; mode 3: light teams
    # (activations loaded straight into registers where eligible); mode 4: light teams with
    # bulk-copied activations
    rng = np.random.default_rng(M * 7 + N)
    x = synth.activations(rng, M, K)
    w = synth.quant_weights(rng, N, K, bits)
    T.tune_set(T.TF_TUNE_MODE, mode)
    try:
        if dual:
            u = synth.quant_weights(rng, N, K, bits)
            g = synth.gamma(rng, K)
            h = T.tf_qmlp_gateup_run(pack(T, w), pack(T, u), dev_bf16(x), gamma=dev_bf16(g), eps=1e-6)
        else:
            y = T.tf_qlinear_run(pack(T, w), dev_bf16(x))
    finally:
        T.tune_set(T.TF_TUNE_MODE, -1)
    if dual:
        ref = oracle.gateup(oracle.bf16_to_f64(x), w, u, oracle.bf16_to_f64(g), 1e-6)
        assert_close(host_f64(h), ref["h"], tol_swiglu(ref["g"], ref["u"], ref["g_abs"], ref["u_abs"]), f"mode {mode}")
    else:
        y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(x), w)
        assert_close(host_f64(y), y_ref, tol_linear(ad), f"mode {mode}")


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("case", ["below_4096", "near_65536", "beyond_65536", "tiny"])
def test_warp_workers_fp16_activation_edges(T, bits, case):
    # the warp workers convert staged activations to fp16 when every value converts
    # exactly (|x| < 65536, finite; for 4-bit codes |x| < 4096) and keep bf16
    # otherwise; fp16 subnormals round
    rng = np.random.default_rng(["below_4096", "near_65536", "beyond_65536", "tiny"].index(case) * 10 + bits)
    M, K, N = 3, 1024, 4096
    xf = rng.standard_normal((M, K)).astype(np.float32)
    if case == "below_4096":
        xf[0, 5], xf[2, 700] = 4080.0, -3968.0  # fp16 path for both code widths
    elif case == "near_65536":
        xf[0, 5], xf[2, 700] = 65280.0, -61440.0  # largest bf16 values below 65536
    elif case == "beyond_65536":
        xf[1, 17] = 131072.0  # the bf16 path for the CTAs staging row 1
    else:
        xf *= 1e-6  # fp16 subnormal range
    x = synth.f32_to_bf16_bits(xf)
    w = synth.quant_weights(rng, N, K, bits)
    T.tune_set(T.TF_TUNE_MODE, 2)
    try:
        y = T.tf_qlinear_run(pack(T, w), dev_bf16(x), out_dtype=torch.float32)
    finally:
        T.tune_set(T.TF_TUNE_MODE, -1)
    y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(x), w)
    assert_close(host_f64(y), y_ref, tol_linear(ad), f"warp workers, {case}, {bits}-bit")


@pytest.mark.parametrize("warps,chunk", [(8, 32), (16, 32), (8, 16), (8, 64)])
@pytest.mark.parametrize("M,K,N,bits,norm", [
    (8, 12800, 2560, 4, False),  # 8 K splits of 25 groups, stream-K cuts inside row blocks
    (1, 12800, 2560, 4, False),
    (3, 2048, 1000, 8, False),   # ragged N, 8-bit codes
    (8, 1024, 4100, 4, True),    # RMSNorm over whole staged rows, ragged last row block
    (1, 1024, 30000, 4, True),   # many whole row blocks per CTA, stored without partials
    (5, 640, 333, 4, False),     # fewer units than CTAs: CTAs capped at one unit each
    (2, 64, 48, 4, True),        # one group a row block
])
def test_streaming_schedule_matches_oracle(T, warps, chunk, M, K, N, bits, norm):
    # the streaming schedule forced on every shape (it is the default only above 8 MB of
    # weights), with a residual and an fp32 output; the workspace is left all-zero
    rng = np.random.default_rng(M * 131 + N + K + warps + chunk)
    x = synth.activations(rng, M, K)
    w = synth.quant_weights(rng, N, K, bits)
    gamma_h = synth.gamma(rng, K) if norm else None
    res_h = synth.activations(rng, M, N)
    qw = pack(T, w)
    T.tune_set(T.TF_TUNE_MODE, 5)
    T.tune_set(T.TF_TUNE_WARPS, warps)
    T.tune_set(T.TF_TUNE_STAGE_GROUPS, chunk)
    try:
        ws = T.workspace(T.tf_qlinear_workspace_bytes(qw, 8))  # sized for the tuned plan
        y = T.tf_qlinear_run(qw, dev_bf16(x), gamma=dev_bf16(gamma_h) if norm else None, eps=1e-6,
                             residual=dev_bf16(res_h), ws=ws, out_dtype=torch.float32)
        torch.cuda.synchronize()
    finally:
        for key in (T.TF_TUNE_MODE, T.TF_TUNE_WARPS, T.TF_TUNE_STAGE_GROUPS):
            T.tune_set(key, -1)
    assert T.tf_workspace_status(ws) == T.TF_OK
    assert int(ws.count_nonzero()) == 0
    xd = oracle.bf16_to_f64(x)
    if norm:
        xd = oracle.rmsnorm(xd, oracle.bf16_to_f64(gamma_h), 1e-6)
    y_ref, ad = oracle.qlinear(xd, w)
    y_ref = y_ref + oracle.bf16_to_f64(res_h)
    tol = tol_linear(ad) + (2.0 ** -8 * np.abs(y_ref) if norm else 0.0)
    assert_close(host_f64(y), y_ref, tol, f"streaming W={warps} CH={chunk}")


@pytest.mark.parametrize("mode", [-1, 1, 2, 3, 4, 5])
@pytest.mark.parametrize("M,K,N,bits,norm", [
    (1, 1024, 3072, 4, False),
    (8, 1024, 3072, 4, True),
    (3, 2048, 1000, 8, False),
    (8, 12800, 2560, 4, False),  # K split: every split rotates its own groups
    (2, 1024, 18992, 4, True),
])
def test_rht_projection_matches_oracle(T, mode, M, K, N, bits, norm):
    # tf_qlinear_run_rht: the input Hadamard transform folded into every staging path
    # (planner's choice, lock-step teams, warp workers, light teams with register-loaded
    # and with bulk-copied activations, streaming), after the RMSNorm when there is one
    rng = np.random.default_rng(600 + M + K + N + bits + mode)
    x = synth.activations(rng, M, K)
    w = synth.quant_weights(rng, N, K, bits)
    signs = synth.rht_signs(rng, K)
    gamma_h = synth.gamma(rng, K) if norm else None
    res_h = synth.activations(rng, M, N)
    qw = pack(T, w)
    T.tune_set(T.TF_TUNE_MODE, mode)
    try:
        ws = T.workspace(T.tf_qlinear_workspace_bytes(qw, 8))
        y = T.tf_qlinear_run_rht(qw, dev_bf16(x), torch.from_numpy(signs).cuda(),
                                 gamma=dev_bf16(gamma_h) if norm else None, eps=1e-6, residual=dev_bf16(res_h),
                                 ws=ws, out_dtype=torch.float32)
        torch.cuda.synchronize()
    finally:
        T.tune_set(T.TF_TUNE_MODE, -1)
    assert T.tf_workspace_status(ws) == T.TF_OK
    xd = oracle.bf16_to_f64(x)
    if norm:
        xd = oracle.rmsnorm(xd, oracle.bf16_to_f64(gamma_h), 1e-6)
    y_ref, ad = oracle.qlinear(oracle.rht(xd, signs), w)
    y_ref = y_ref + oracle.bf16_to_f64(res_h)
    assert_close(host_f64(y), y_ref, tol_linear(ad), f"rht, mode {mode}")


def test_rht_with_zero_signs_is_not_the_plain_projection(T):
    # control: with the transform the result differs from the plain call on the same
    # inputs (the rotation is applied), and equals it after rotating x on the host
    rng = np.random.default_rng(650)
    M, K, N = 2, 1024, 512
    x = synth.activations(rng, M, K)
    w = synth.quant_weights(rng, N, K, 4)
    signs = np.zeros(K // 8, np.uint8)
    qw = pack(T, w)
    y_rht = host_f64(T.tf_qlinear_run_rht(qw, dev_bf16(x), torch.from_numpy(signs).cuda(), out_dtype=torch.float32))
    y_plain = host_f64(T.tf_qlinear_run(qw, dev_bf16(x), out_dtype=torch.float32))
    assert np.abs(y_rht - y_plain).max() > 1.0
    xr = synth.f32_to_bf16_bits(oracle.rht(oracle.bf16_to_f64(x), signs).astype(np.float32))
    y_host = host_f64(T.tf_qlinear_run(qw, dev_bf16(xr), out_dtype=torch.float32))
    _, ad = oracle.qlinear(oracle.rht(oracle.bf16_to_f64(x), signs), w)
    assert_close(y_rht, y_host, tol_linear(ad), "rht on device vs on host")
