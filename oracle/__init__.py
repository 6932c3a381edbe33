"""fp64 CPU oracle for the 4/8-bit group-quantised decode projection.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` are the only
callers. Nothing in the ``skinny_gemm_bit_gb300`` package imports this module,
and this module imports nothing from that package.

The arithmetic lives in ``oracle.c`` (plain loops in double precision); this
file only marshals numpy arrays and composes the C primitives in the order the
pages describe:

* ``qlinear``   -- y = x . dequant(W)^T for MLX affine weights (uzu page,
  "Internals 1" table, weight_matrix row; TensorFold page, box smoke-test
  table, "4-bit group 64").
* ``gateup``    -- RMSNorm folded ahead of gate and up, SwiGLU epilogue
  (Husky page, "Four implementation elements of MSI").
* ``moe``       -- per-row top-k expert routing, SwiGLU experts, weighted sum
  (uzu page, "Internals 1" table, mlp row: MixtureOfExperts + routing).
* ``decode_step`` -- one decoder step as four projections per layer and a
  tied readout (Husky page, "Four implementation elements of MSI": one layer
  is four consecutive kernels; uzu page, "Internals 1": Qwen3-0.6B dims,
  28 layers, model_dim 1024, hidden 3072, vocab 151,936, tied embedding).

Weights are passed as dicts with keys ``wq`` (uint32 [N, K*bits/32]),
``scales`` / ``biases`` (uint16 bf16 bits [N, K/64]), ``N``, ``K``, ``bits``.
Stacks of experts use a leading batch axis on the three arrays. NVFP4 weights
(TensorFold page, "qualified" model table: NVFP4 checkpoints; format as read in
``oracle.c``) are dicts with ``code`` = "nvfp4", ``codes`` (uint8 [N, K/2], even
column in the low nibble), ``scales`` (uint8 E4M3 [N, K/16]), ``gscale`` (fp32),
``N``, ``K``; ``dequant``, ``qlinear`` and ``gateup`` accept them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
GROUP = 64

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/liboracle.so with gcc (-O2, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                           "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    lib.oracle_unpack.argtypes = [P, I64, I64, I, P]
    lib.oracle_unpack.restype = I
    lib.oracle_dequant.argtypes = [P, P, P, I64, I64, I, I, P]
    lib.oracle_dequant.restype = I
    lib.oracle_qlinear.argtypes = [P, I64, I64, P, P, P, I64, I64, I, I, P, P]
    lib.oracle_qlinear.restype = I
    lib.oracle_rmsnorm.argtypes = [P, I64, I64, P, ctypes.c_double, P]
    lib.oracle_rmsnorm.restype = None
    lib.oracle_swiglu.argtypes = [P, P, I64, P]
    lib.oracle_swiglu.restype = None
    lib.oracle_topk_softmax.argtypes = [P, I64, I64, I64, P, P]
    lib.oracle_topk_softmax.restype = I
    lib.oracle_rht.argtypes = [P, I64, I64, P, I64, P]
    lib.oracle_rht.restype = I
    D = ctypes.c_double
    lib.oracle_e2m1.argtypes = [I]
    lib.oracle_e2m1.restype = D
    lib.oracle_e4m3.argtypes = [I]
    lib.oracle_e4m3.restype = D
    lib.oracle_nvfp4_dequant.argtypes = [P, P, D, I64, I64, P]
    lib.oracle_nvfp4_dequant.restype = I
    lib.oracle_nvfp4_qlinear.argtypes = [P, I64, I64, P, P, D, I64, I64, P, P]
    lib.oracle_nvfp4_qlinear.restype = I
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# primitives
# ----------------------------------------------------------------------------

def unpack(wq, N: int, K: int, bits: int) -> np.ndarray:
    """q[n][k] as uint8 [N, K]; element j of a word is bits [bits*j, bits*j+bits)."""
    wq = _c(wq, np.uint32)
    q = np.empty((N, K), dtype=np.uint8)
    rc = _load().oracle_unpack(_ptr(wq), N, K, bits, _ptr(q))
    if rc:
        raise ValueError(f"oracle_unpack rejected N={N} K={K} bits={bits}")
    return q


def is_nvfp4(w: dict) -> bool:
    return w.get("code") == "nvfp4"


def e2m1(code: int) -> float:
    """Value of a 4-bit E2M1 code (NVFP4 element)."""
    return _load().oracle_e2m1(int(code))


def e4m3(code: int) -> float:
    """Value of an E4M3 byte (NVFP4 block scale); NaN for S.1111.111."""
    return _load().oracle_e4m3(int(code))


def nvfp4_dequant(w: dict) -> np.ndarray:
    """w[n][k] = gscale * e4m3(scales[n][k/16]) * e2m1(q[n][k]) in float64 [N, K]."""
    N, K = w["N"], w["K"]
    out = np.empty((N, K), dtype=np.float64)
    rc = _load().oracle_nvfp4_dequant(_ptr(_c(w["codes"], np.uint8)), _ptr(_c(w["scales"], np.uint8)),
                                      float(np.float32(w["gscale"])), N, K, _ptr(out))
    if rc:
        raise ValueError("oracle_nvfp4_dequant rejected the weights")
    return out


def dequant(w: dict) -> np.ndarray:
    """w[n][k] = scale*q + bias in float64 [N, K] (NVFP4 weights: ``nvfp4_dequant``)."""
    if is_nvfp4(w):
        return nvfp4_dequant(w)
    N, K, bits = w["N"], w["K"], w["bits"]
    out = np.empty((N, K), dtype=np.float64)
    rc = _load().oracle_dequant(_ptr(_c(w["wq"], np.uint32)), _ptr(_c(w["scales"], np.uint16)),
                                _ptr(_c(w["biases"], np.uint16)), N, K, bits, GROUP, _ptr(out))
    if rc:
        raise ValueError("oracle_dequant rejected the weights")
    return out


def qlinear(x, w: dict):
    """(y, absdot): y[m][n] = sum_k x[m][k] w[n][k]; absdot = sum_k |x w|.

    ``x`` is float64 [M, K] (use ``bf16_to_f64`` for bf16 activations).
    """
    x = _c(np.atleast_2d(x), np.float64)
    M, K = x.shape
    if K != w["K"]:
        raise ValueError(f"x has K={K}, weights have K={w['K']}")
    N = w["N"]
    y = np.empty((M, N), dtype=np.float64)
    ad = np.empty((M, N), dtype=np.float64)
    if is_nvfp4(w):
        rc = _load().oracle_nvfp4_qlinear(_ptr(x), K, M, _ptr(_c(w["codes"], np.uint8)),
                                          _ptr(_c(w["scales"], np.uint8)), float(np.float32(w["gscale"])),
                                          N, K, _ptr(y), _ptr(ad))
        if rc:
            raise ValueError("oracle_nvfp4_qlinear rejected the weights")
        return y, ad
    rc = _load().oracle_qlinear(_ptr(x), K, M, _ptr(_c(w["wq"], np.uint32)),
                                _ptr(_c(w["scales"], np.uint16)), _ptr(_c(w["biases"], np.uint16)),
                                N, K, w["bits"], GROUP, _ptr(y), _ptr(ad))
    if rc:
        raise ValueError("oracle_qlinear rejected the weights")
    return y, ad


def rmsnorm(x, gamma, eps: float) -> np.ndarray:
    """xn = x / sqrt(mean(x^2) + eps) * gamma, per row, in float64."""
    x = _c(np.atleast_2d(x), np.float64)
    gamma = _c(gamma, np.float64)
    M, K = x.shape
    out = np.empty_like(x)
    _load().oracle_rmsnorm(_ptr(x), M, K, _ptr(gamma), float(eps), _ptr(out))
    return out


def rht(x, signs, block: int = 64) -> np.ndarray:
    """Input randomized Hadamard transform, float64: per block of `block` columns,
    H (d * x) / sqrt(block), H Sylvester-ordered, d[k] = -1 where bit k of the
    LSB-first bit vector `signs` (uint8 [K / 8]) is set (uzu page, "Internals 1"
    table, linear row: input RHT)."""
    x = _c(np.atleast_2d(x), np.float64)
    M, K = x.shape
    signs = _c(signs, np.uint8)
    if signs.size * 8 < K:
        raise ValueError("signs must hold K bits")
    out = np.empty_like(x)
    if _load().oracle_rht(_ptr(x), M, K, _ptr(signs), block, _ptr(out)):
        raise ValueError(f"block {block} must be a power of two dividing K={K}")
    return out


def swiglu(g, u) -> np.ndarray:
    """silu(g) * u elementwise, float64."""
    g = _c(g, np.float64)
    u = _c(u, np.float64)
    if g.shape != u.shape:
        raise ValueError("gate and up shapes differ")
    out = np.empty_like(g)
    _load().oracle_swiglu(_ptr(g), _ptr(u), g.size, _ptr(out))
    return out


def topk_softmax(logits, top_k: int):
    """(idx int32 [M, k], w float64 [M, k]) for fp32 router logits [M, E]."""
    logits = _c(np.atleast_2d(logits), np.float32)
    M, E = logits.shape
    idx = np.empty((M, top_k), dtype=np.int32)
    w = np.empty((M, top_k), dtype=np.float64)
    rc = _load().oracle_topk_softmax(_ptr(logits), M, E, top_k, _ptr(idx), _ptr(w))
    if rc:
        raise ValueError(f"oracle_topk_softmax rejected top_k={top_k} E={E}")
    return idx, w


# ----------------------------------------------------------------------------
# compositions
# ----------------------------------------------------------------------------

def expert(w: dict, e: int) -> dict:
    """The e-th matrix of a stacked [E, ...] weight dict (NVFP4 stacks: codes, block
    scales and one global scale per expert)."""
    if is_nvfp4(w):
        return {"code": "nvfp4", "codes": w["codes"][e], "scales": w["scales"][e],
                "gscale": np.float32(np.asarray(w["gscale"]).reshape(-1)[e]), "N": w["N"], "K": w["K"]}
    return {"wq": w["wq"][e], "scales": w["scales"][e], "biases": w["biases"][e],
            "N": w["N"], "K": w["K"], "bits": w["bits"]}


def gateup(x, gate: dict, up: dict, gamma=None, eps: float = 1e-6) -> dict:
    """RMSNorm (optional) -> gate, up -> h = silu(gate) * up.

    Returns every intermediate the parity tolerance needs: xn, g, u, h and the
    absdot sums of both projections.
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    xn = rmsnorm(x, gamma, eps) if gamma is not None else x
    g, g_abs = qlinear(xn, gate)
    u, u_abs = qlinear(xn, up)
    return {"xn": xn, "g": g, "u": u, "g_abs": g_abs, "u_abs": u_abs, "h": swiglu(g, u)}


def moe(x, logits, gate: dict, up: dict, down: dict, top_k: int) -> dict:
    """Per-row top-k routing, per-expert SwiGLU MLP, weighted sum over slots.

    y[m] = sum_j w[m][j] * down_e(silu(gate_e x[m]) * up_e x[m]), e = idx[m][j].
    Also returns the per-(m, j) expert intermediates for the tolerance.
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    idx, wts = topk_softmax(logits, top_k)
    M = x.shape[0]
    H = down["N"]
    y = np.zeros((M, H), dtype=np.float64)
    slots = []
    for m in range(M):
        row = []
        for j in range(top_k):
            e = int(idx[m, j])
            gu = gateup(x[m:m + 1], expert(gate, e), expert(up, e))
            o, o_abs = qlinear(gu["h"], expert(down, e))
            y[m] += wts[m, j] * o[0]
            row.append({"e": e, "g": gu["g"][0], "u": gu["u"][0], "g_abs": gu["g_abs"][0],
                        "u_abs": gu["u_abs"][0], "h": gu["h"][0], "o": o[0], "o_abs": o_abs[0]})
        slots.append(row)
    return {"idx": idx, "w": wts, "y": y, "slots": slots}


def decode_step(x, layers, final_norm, readout: dict, q_dim: int, eps: float = 1e-6,
                readout_rows=None) -> dict:
    """One decoder step through the projections only (attention excluded).

    Per layer (four projections, in order):
      qkv = rmsnorm(h, attn_norm) . Wqkv^T          (q | k | v concatenated)
      h   = h + qkv[:, :q_dim] . Wo^T               (q stands in for attention)
      a   = silu(rmsnorm(h, mlp_norm) . Wg^T) * (rmsnorm(h, mlp_norm) . Wu^T)
      h   = h + a . Wd^T
    then logits = rmsnorm(h, final_norm) . Wreadout^T.

    ``layers`` is a list of dicts with keys qkv, o, gate, up, down (weight dicts)
    and attn_norm, mlp_norm (float64 gammas). ``readout_rows`` optionally limits
    the readout to a subset of vocabulary rows (index array), for large vocabularies.
    Returns the per-stage values and their absdot sums.
    """
    h = np.atleast_2d(np.asarray(x, dtype=np.float64))
    stages = []
    for L in layers:
        xn = rmsnorm(h, L["attn_norm"], eps)
        qkv, qkv_abs = qlinear(xn, L["qkv"])
        q = qkv[:, :q_dim]
        o, o_abs = qlinear(q, L["o"])
        h1 = h + o
        gu = gateup(h1, L["gate"], L["up"], L["mlp_norm"], eps)
        d, d_abs = qlinear(gu["h"], L["down"])
        h2 = h1 + d
        stages.append({"xn": xn, "qkv": qkv, "qkv_abs": qkv_abs, "o": o, "o_abs": o_abs,
                       "h1": h1, "gu": gu, "d": d, "d_abs": d_abs, "h2": h2})
        h = h2
    xf = rmsnorm(h, final_norm, eps)
    ro = readout
    if readout_rows is not None:
        rows = np.asarray(readout_rows)
        if is_nvfp4(readout):
            ro = dict(readout, codes=readout["codes"][rows], scales=readout["scales"][rows], N=len(rows))
        else:
            ro = {"wq": readout["wq"][rows], "scales": readout["scales"][rows],
                  "biases": readout["biases"][rows], "N": len(rows), "K": readout["K"],
                  "bits": readout["bits"]}
    logits, l_abs = qlinear(xf, ro)
    return {"stages": stages, "h": h, "xf": xf, "logits": logits, "logits_abs": l_abs}
