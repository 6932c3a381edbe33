"""tf_qlinear_run_noalloc (scratch in the library's fixed device array) against
tf_qlinear_run (caller workspace) and the fp64 oracle.

Collected last on purpose: it must pass both alone in a fresh process and after
every other test has run in the same process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, dev_bf16, host_f64, pack, tol_linear
from skinny_gemm_bit_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    from skinny_gemm_bit_gb300 import build
    build.build()
    from skinny_gemm_bit_gb300 import tfq
    return tfq


# (M, K, N, bits, rmsnorm + residual): the wide shape splits K across CTAs, so its
# counters and partial slots live in the fixed array and must come back clean
CASES = [
    (1, 1024, 3072, 4, False),
    (8, 12800, 2560, 4, False),
    (1, 12800, 2560, 4, False),
    (3, 2048, 1000, 8, True),
]


@pytest.mark.parametrize("M,K,N,bits,norm", CASES)
def test_noalloc_matches_workspace_call_twice_in_a_row(T, M, K, N, bits, norm):
    cfg = synth.single_projection(seed=7000 + M + N, M=M, K=K, N=N, bits=bits)
    w = pack(T, cfg["w"])
    x = dev_bf16(cfg["x"])
    rng = np.random.default_rng(7100 + M)
    gamma = res = None
    if norm:
        gamma_h = synth.gamma(rng, K)
        res_h = synth.activations(rng, M, N)
        gamma, res = dev_bf16(gamma_h), dev_bf16(res_h)
    y_ws = T.tf_qlinear_run(w, x, gamma=gamma, eps=1e-6, residual=res)
    outs = []
    for _ in range(2):
        y = T.tf_qlinear_run_noalloc(w, x, gamma=gamma, eps=1e-6, residual=res)
        torch.cuda.synchronize()
        outs.append(host_f64(y))
    ref_ws = host_f64(y_ws)
    if norm:
        xn = oracle.rmsnorm(oracle.bf16_to_f64(cfg["x"]), oracle.bf16_to_f64(gamma_h), 1e-6)
        y_ref, ad = oracle.qlinear(xn, cfg["w"])
        y_ref = y_ref + oracle.bf16_to_f64(res_h)
        tol = tol_linear(ad) + 2.0 ** -8 * np.abs(y_ref)
    else:
        y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(cfg["x"]), cfg["w"])
        tol = tol_linear(ad)
    for i, y in enumerate(outs):
        # same kernels and launch plan as the workspace call: the results agree within
        # the projection tolerance (in practice byte for byte), and with the oracle
        assert_close(y, ref_ws, tol, f"noalloc call {i} vs tf_qlinear_run, M={M} K={K} N={N}")
        assert_close(y, y_ref, tol, f"noalloc call {i} vs oracle, M={M} K={K} N={N}")
    # no device-side failure was recorded in the fixed array by these calls
    assert T.tf_qlinear_noalloc_status() == T.TF_OK


def test_noalloc_refuses_a_shape_beyond_the_fixed_scratch(T):
    # K=12800 splits into 4 slices; with N=151936 the partial slots need ~19 MB, more
    # than the 4 MiB array: refused on the host before anything is enqueued (the
    # descriptor's data pointer is never read)
    holder = torch.zeros(64, dtype=torch.uint8, device="cuda")
    d = T.tf_qweight()
    d.magic, d.version, d.bits, d.group = T.TF_QWEIGHT_MAGIC, T.TF_PACK_VERSION, 4, 64
    d.batch, d.N, d.K = 1, 151936, 12800
    d.n_pad = (d.N + 15) // 16 * 16
    d.tile_bytes = 576
    d.matrix_bytes = d.n_pad // 16 * (d.K // 64) * 576
    d.data = holder.data_ptr()
    assert T.lib().tf_qlinear_workspace_bytes(ctypes.byref(d), 8) > 4 << 20
    x = torch.zeros((8, 12800), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((8, 151936), dtype=torch.bfloat16, device="cuda")
    rc = T.lib().tf_qlinear_run_noalloc(ctypes.byref(d), ctypes.c_void_p(x.data_ptr()), 12800, 8, None, 1e-6, None,
                                        ctypes.c_void_p(y.data_ptr()), T.TF_DTYPE_BF16, 0, None)
    assert rc == T.TF_E_WORKSPACE_TOO_SMALL
    msg = T.lib().tf_last_error().decode()
    assert "4194304" in msg and "tf_qlinear_run" in msg, msg


@pytest.mark.parametrize("M,K,N", [(8, 12800, 2560), (1, 1024, 3072)])
def test_noalloc_nvfp4_matches_workspace_call(T, M, K, N):
    # NVFP4 descriptors through the fixed-array entry point: the same kernels, the same bits
    rng = np.random.default_rng(7200 + M)
    w = synth.nvfp4_weights(rng, N, K)
    x = dev_bf16(synth.activations(rng, M, K))
    qw = T.tf_qlinear_pack_nvfp4(w["codes"], w["scales"], float(w["gscale"]))
    y_ws = T.tf_qlinear_run(qw, x)
    y = T.tf_qlinear_run_noalloc(qw, x)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_ws.view(torch.int16))


def test_noalloc_status_reports_a_timeout_and_clears_the_array(T):
    # a bounded wait that nothing satisfies, aimed at the fixed array's status word (a
    # 1 ms limit: the kernel gives up and returns, the GPU stays usable), then the
    # status query reports it once, puts the array back to zero, and the next
    # split-K projection through the array matches the oracle
    T.tf_selftest_wait_timeout(None, 1_000_000)
    assert T.tf_qlinear_noalloc_status() == T.TF_E_TIMEOUT
    assert "cleared" in T.lib().tf_last_error().decode()
    assert T.tf_qlinear_noalloc_status() == T.TF_OK
    cfg = synth.single_projection(seed=7300, M=8, K=12800, N=2560, bits=4)
    w = pack(T, cfg["w"])
    y = T.tf_qlinear_run_noalloc(w, dev_bf16(cfg["x"]))
    torch.cuda.synchronize()
    y_ref, ad = oracle.qlinear(oracle.bf16_to_f64(cfg["x"]), cfg["w"])
    assert_close(host_f64(y), y_ref, tol_linear(ad), "noalloc call after a cleared timeout")
    assert T.tf_qlinear_noalloc_status() == T.TF_OK


def test_noalloc_errors_name_the_noalloc_entry_point(T):
    # an argument error found by the shared projection path is reported under this
    # entry point's name, not tf_qlinear_run's
    cfg = synth.single_projection(seed=7400, M=1, K=1024, N=64, bits=4)
    w = pack(T, cfg["w"])
    x = torch.zeros((1, 1024), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((1, 64), dtype=torch.bfloat16, device="cuda")
    rc = T.lib().tf_qlinear_run_noalloc(ctypes.byref(w.desc), ctypes.c_void_p(x.data_ptr()), 1024, 1, None, 1e-6,
                                        None, ctypes.c_void_p(y.data_ptr()), 7, 0, None)  # 7: no such y dtype
    assert rc == T.TF_E_INVALID_ARG
    assert T.lib().tf_last_error().decode().startswith("tf_qlinear_run_noalloc:")
