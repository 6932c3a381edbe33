"""Seeded synthetic inputs for the quantised decode projection workloads.

This module is the only code shared by the CUDA-path tests, the oracle tests
and the benchmark. It draws random numbers and lays them out in the MLX input
format; it holds none of the projection arithmetic (no unpacking, no
dequantisation, no products).

Recipes (numpy ``default_rng`` / PCG64, draws in the order written here):

* activations x ~ N(0, 1), drawn in fp32, rounded to bf16 (round to nearest even);
* 4-bit codes q uniform in [0, 15], packed 8 per uint32 along K, element j of a
  word in bits [4j, 4j+4); uniform random 32-bit words are exactly this;
* 8-bit codes q uniform in [0, 255], 4 per uint32, element j in bits [8j, 8j+8);
* per-64-K-group scale ~ |N(0, 0.02)| (4-bit) or |N(0, 0.02)| / 16 (8-bit, so
  that the 8-bit layer spans the same weight range as the 4-bit one), rounded
  to bf16; bias = -2^(bits-1) * scale + N(0, 0.002), formed in fp32 from the
  bf16 scale, then rounded to bf16;
* RMSNorm gamma ~ N(1, 0.1) in bf16; router logits ~ N(0, 1) in fp32.
* NVFP4 weights: code bytes uniform in [0, 255] (two E2M1 codes each, every code
  equally likely, -0 included); block-scale bytes positive E4M3 with exponent field
  uniform in [4, 11] and mantissa uniform in [0, 7] (0.125 .. 15), one block in 64
  replaced by an edge byte (0x00 zero, 0x01 smallest subnormal, 0x07 largest
  subnormal, 0x7E largest normal, 448); global scale 0.004 (fp32).
"""
from __future__ import annotations

import numpy as np

GROUP = 64


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        rounded = np.where(nan, np.uint16(0x7FC0), rounded)
    return rounded


def bf16_bits_to_f32(b) -> np.ndarray:
    """bf16 bit patterns (uint16) to fp32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def pack_codes(q, bits: int) -> np.ndarray:
    """Pack integer codes [..., K] into uint32 words along K, LSB-first."""
    q = np.asarray(q)
    per = 32 // bits
    K = q.shape[-1]
    if K % per:
        raise ValueError("K must be a multiple of the codes per word")
    qw = q.astype(np.uint32).reshape(*q.shape[:-1], K // per, per)
    out = np.zeros(qw.shape[:-1], dtype=np.uint32)
    for j in range(per):
        out |= qw[..., j] << np.uint32(bits * j)
    return out


def activations(rng, M: int, K: int) -> np.ndarray:
    """x ~ N(0, 1) as bf16 bits [M, K]."""
    return f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))


def gamma(rng, K: int) -> np.ndarray:
    """RMSNorm weight ~ N(1, 0.1) as bf16 bits [K]."""
    return f32_to_bf16_bits(1.0 + 0.1 * rng.standard_normal(K, dtype=np.float32))


def rht_signs(rng, K: int) -> np.ndarray:
    """Random +-1 signs of an input Hadamard transform as K bits (uint8 [K / 8],
    least-significant bit first, bit set = -1), uniform and independent."""
    return rng.integers(0, 256, size=(K + 7) // 8, dtype=np.uint8)


def router_logits(rng, M: int, E: int) -> np.ndarray:
    """Router logits ~ N(0, 1), fp32 [M, E]."""
    return rng.standard_normal((M, E), dtype=np.float32)


def quant_weights(rng, N: int, K: int, bits: int = 4, batch: int | None = None) -> dict:
    """Random MLX affine weights: wq uint32 [(B,) N, K*bits/32], scales/biases bf16 [(B,) N, K/64]."""
    if bits not in (4, 8):
        raise ValueError("bits must be 4 or 8")
    if K % GROUP:
        raise ValueError("K must be a multiple of 64")
    lead = () if batch is None else (batch,)
    words = K * bits // 32
    wq = rng.integers(0, 2**32, size=lead + (N, words), dtype=np.uint32)
    sigma = 0.02 if bits == 4 else 0.02 / 16.0
    s32 = np.abs(rng.standard_normal(lead + (N, K // GROUP), dtype=np.float32)) * np.float32(sigma)
    scales = f32_to_bf16_bits(s32)
    noise = rng.standard_normal(lead + (N, K // GROUP), dtype=np.float32) * np.float32(0.002)
    b32 = np.float32(-(2 ** (bits - 1))) * bf16_bits_to_f32(scales) + noise
    biases = f32_to_bf16_bits(b32)
    return {"wq": wq, "scales": scales, "biases": biases, "N": N, "K": K, "bits": bits}


def nvfp4_weights(rng, N: int, K: int, batch: int | None = None) -> dict:
    """Random NVFP4 weights: codes uint8 [(B,) N, K/2] (even column in the low nibble),
    E4M3 block scales uint8 [(B,) N, K/16], fp32 global scale (a stack of B experts: one
    per expert, 0.004 times a power of two from 1/2 to 2, so each expert's differs)."""
    if K % GROUP:
        raise ValueError("K must be a multiple of 64")
    lead = () if batch is None else (batch,)
    codes = rng.integers(0, 256, size=lead + (N, K // 2), dtype=np.uint8)
    e = rng.integers(4, 12, size=lead + (N, K // 16), dtype=np.uint8)
    m = rng.integers(0, 8, size=lead + (N, K // 16), dtype=np.uint8)
    scales = (e << 3) | m
    edge = rng.integers(0, 64, size=lead + (N, K // 16)) == 0
    pick = np.array([0x00, 0x01, 0x07, 0x7E], dtype=np.uint8)[rng.integers(0, 4, size=lead + (N, K // 16))]
    scales = np.where(edge, pick, scales).astype(np.uint8)
    if batch is None:
        gscale = np.float32(0.004)
    else:
        gscale = (np.float32(0.004) * np.exp2(rng.integers(-1, 2, size=batch)).astype(np.float32)).astype(np.float32)
    return {"code": "nvfp4", "codes": codes, "scales": scales, "gscale": gscale, "N": N, "K": K}


def concat_rows(*ws) -> dict:
    """Stack weight dicts along N (e.g. q | k | v into one projection)."""
    return {"wq": np.concatenate([w["wq"] for w in ws], axis=-2),
            "scales": np.concatenate([w["scales"] for w in ws], axis=-2),
            "biases": np.concatenate([w["biases"] for w in ws], axis=-2),
            "N": sum(w["N"] for w in ws), "K": ws[0]["K"], "bits": ws[0]["bits"]}


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------

def nvfp4_projection(seed: int, M: int, K: int, N: int) -> dict:
    """One NVFP4 projection: activations, then the weights (``nvfp4_weights``)."""
    rng = np.random.default_rng(seed)
    x = activations(rng, M, K)
    return {"x": x, "w": nvfp4_weights(rng, N, K)}


def single_projection(seed: int = 0, M: int = 1, K: int = 1024, N: int = 3072, bits: int = 4) -> dict:
    """One 4-bit projection (default: M=1, K=1024, N=3072, seed 0)."""
    rng = np.random.default_rng(seed)
    x = activations(rng, M, K)
    w = quant_weights(rng, N, K, bits)
    return {"x": x, "w": w}


def fused_gateup(seed: int = 1, M: int = 8, K: int = 1024, N: int = 3072, bits: int = 4) -> dict:
    """RMSNorm + gate/up SwiGLU (default: K=1024, N=3072 per matrix, eps 1e-6)."""
    rng = np.random.default_rng(seed)
    x = activations(rng, M, K)
    g = gamma(rng, K)
    gate = quant_weights(rng, N, K, bits)
    up = quant_weights(rng, N, K, bits)
    return {"x": x, "gamma": g, "eps": 1e-6, "gate": gate, "up": up}


def wide_verify(seed: int = 2, M: int = 8, K: int = 12800, N: int = 2560, bits: int = 4) -> dict:
    """Down projection of a ~4B dense model (default: M=8, K=12800, N=2560)."""
    return single_projection(seed=seed, M=M, K=K, N=N, bits=bits)


def decoder(seed: int = 3, n_layers: int = 28, d_model: int = 1024, d_ff: int = 3072,
            n_q_heads: int = 16, n_kv_heads: int = 8, head_dim: int = 128,
            vocab: int = 151936, M: int = 1, bits: int = 4, code: str = "mlx") -> dict:
    """Random weights of a dense decoder's projections plus a tied readout (MLX affine
    codes of `bits`, or NVFP4 with code="nvfp4")."""
    rng = np.random.default_rng(seed)
    q_dim = n_q_heads * head_dim
    kv_dim = n_kv_heads * head_dim
    x = activations(rng, M, d_model)

    def weights(N, K):
        return nvfp4_weights(rng, N, K) if code == "nvfp4" else quant_weights(rng, N, K, bits)

    layers = []
    for _ in range(n_layers):
        layers.append({
            "attn_norm": gamma(rng, d_model),
            "qkv": weights(q_dim + 2 * kv_dim, d_model),
            "o": weights(d_model, q_dim),
            "mlp_norm": gamma(rng, d_model),
            "gate": weights(d_ff, d_model),
            "up": weights(d_ff, d_model),
            "down": weights(d_model, d_ff),
        })
    final_norm = gamma(rng, d_model)
    readout = weights(vocab, d_model)
    return {"x": x, "layers": layers, "final_norm": final_norm, "readout": readout,
            "dims": {"n_layers": n_layers, "d_model": d_model, "d_ff": d_ff, "q_dim": q_dim,
                     "kv_dim": kv_dim, "vocab": vocab}, "eps": 1e-6}


def moe_layer(seed: int = 4, M: int = 8, E: int = 128, top_k: int = 8, hidden: int = 2048,
              inter: int = 768, bits: int = 4, code: str = "mlx") -> dict:
    """MoE layer: router logits, per-expert gate/up [E, inter, hidden], down [E, hidden, inter]
    (MLX affine codes of `bits`, or NVFP4 experts with code="nvfp4")."""
    rng = np.random.default_rng(seed)
    x = activations(rng, M, hidden)
    logits = router_logits(rng, M, E)

    def weights(N, K):
        return nvfp4_weights(rng, N, K, batch=E) if code == "nvfp4" else quant_weights(rng, N, K, bits, batch=E)

    gate = weights(inter, hidden)
    up = weights(inter, hidden)
    down = weights(hidden, inter)
    return {"x": x, "logits": logits, "gate": gate, "up": up, "down": down, "top_k": top_k}
