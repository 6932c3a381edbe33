"""Helpers shared by the GPU parity tests: device transfer and the tolerances.

Tolerances (all derived from the stated bound for one projection,
|y - y_ref| <= 1e-2 * sum_k |x_k w_k| + 1e-3, with x the oracle's own input):

* projection:            EPS * absdot + ATOL
* with a residual added: + the residual's own bound (when it is an earlier
                          output) + 2^-8 |y_ref| for the final bf16 rounding
* SwiGLU h = silu(g) u:  |silu'| <= 1.1, so
                          1.1 dg (|u| + du) + |silu(g)| du + 2^-8 |h| + ATOL
                          with dg = EPS S_g, du = EPS S_u
* MoE y = sum_j w_j o_j: sum_j [ |dw_j| |o_j| + w_j (EPS S_o + sum_k tol_h,k |d_k| + ATOL) ] + 2^-8 |y| + ATOL
"""
import numpy as np
import torch

import oracle

EPS = 1e-2
ATOL = 1e-3
BF16_REL = 2.0 ** -8
# tight bounds for fp32 outputs (derivation and measurements in test_gpu_tight_bounds.py)
PLAIN_TIGHT = 2.0 ** -14
NORM_TIGHT = 2.0 ** -9 + 2.0 ** -14
TINY = 1e-7


def dev_bf16(u16) -> torch.Tensor:
    """bf16 bit patterns (numpy uint16) -> torch.bfloat16 on the GPU."""
    a = np.ascontiguousarray(u16, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(a).cuda().view(torch.bfloat16)


def dev_f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def silu(g):
    return g / (1.0 + np.exp(-np.clip(g, -700, 700)))


def tol_linear(absdot):
    return EPS * absdot + ATOL


def tol_swiglu(g, u, g_abs, u_abs, eps=EPS, atol=ATOL):
    dg, du = eps * g_abs, eps * u_abs
    h = silu(g) * u
    return 1.1 * dg * (np.abs(u) + du) + np.abs(silu(g)) * du + BF16_REL * np.abs(h) + atol


def assert_close(y, ref, tol, what=""):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    err = np.abs(y - ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - tol, -np.inf)), y.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {y.size} outside tolerance; worst at {i}: "
                             f"gpu={y[i]!r} ref={ref[i]!r} err={err[i]:.3g} tol={tol[i]:.3g}")


def pack(T, w: dict):
    if w.get("code") == "nvfp4":
        return T.tf_qlinear_pack_nvfp4(w["codes"], w["scales"], w["gscale"])
    return T.tf_qlinear_pack(w["wq"], w["scales"], w["biases"], w["bits"])


def moe_tolerance(ref: dict, down: dict, w_gpu: np.ndarray, eps=EPS, atol=ATOL):
    """Bound on |y_gpu - y_ref| for the MoE layer (see module docstring); eps and atol are
    the per-projection bound's relative and absolute terms."""
    M, k = ref["idx"].shape
    H = ref["y"].shape[1]
    tol = np.zeros((M, H))
    for m in range(M):
        for j in range(k):
            s = ref["slots"][m][j]
            tol_h = tol_swiglu(s["g"], s["u"], s["g_abs"], s["u_abs"], eps, atol)
            _, prop = oracle.qlinear(tol_h[None, :], oracle.expert(down, s["e"]))
            dw = abs(float(w_gpu[m, j]) - ref["w"][m, j])
            tol[m] += dw * np.abs(s["o"]) + ref["w"][m, j] * (eps * s["o_abs"] + prop[0] + atol)
    return tol + BF16_REL * np.abs(ref["y"]) + atol
