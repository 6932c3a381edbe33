"""Pins for the fp64 oracle against facts that do not come from the oracle itself.

Each test fixes one property by a closed form, a hand-worked case, an
invariant, explicit bit patterns, or a textbook routine, chosen so that a
plausible mistake (a dropped term, wrong sign, wrong nibble order, transposed
operand, wrong tie-break) fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from skinny_gemm_bit_gb300 import synth

ONE = 0x3F80  # bf16 1.0


def bf16(v):
    return synth.f32_to_bf16_bits(np.asarray(v, dtype=np.float32))


def weights(wq, scales, biases, N, K, bits):
    return {"wq": np.asarray(wq, np.uint32), "scales": np.asarray(scales, np.uint16),
            "biases": np.asarray(biases, np.uint16), "N": N, "K": K, "bits": bits}


# ---------------------------------------------------------------- unpack order

def test_unpack_4bit_explicit_words():
    # element j of a word sits in bits [4j, 4j+4): 0x76543210 holds 0..7 in order
    wq = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    q = oracle.unpack(wq, 1, 16, 4)
    assert q.tolist() == [list(range(16))]


def test_unpack_8bit_explicit_words():
    wq = np.array([[0x03020100, 0xFFFEFDFC]], dtype=np.uint32)
    q = oracle.unpack(wq, 1, 8, 8)
    assert q.tolist() == [[0, 1, 2, 3, 252, 253, 254, 255]]


def test_unpack_rows_are_independent():
    wq = np.array([[0x11111111], [0x22222222], [0xF0F0F0F0]], dtype=np.uint32)
    q = oracle.unpack(wq, 3, 8, 4)
    assert q.tolist() == [[1] * 8, [2] * 8, [0, 15] * 4]


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("c", [0, 1, 7, 15])
def test_constant_code_unit_scale_ones(c):
    # q = c everywhere, s = 1, b = 0, x = 1  ->  y = K * c exactly
    N, K = 5, 256
    wq = np.full((N, K // 8), c * 0x11111111, dtype=np.uint32)
    w = weights(wq, np.full((N, K // 64), ONE), np.zeros((N, K // 64)), N, K, 4)
    y, ad = oracle.qlinear(np.ones((1, K)), w)
    assert np.all(y == K * c)
    assert np.all(ad == K * c)


def test_bias_only():
    # s = 0, b = beta  ->  y = beta * sum(x)
    N, K = 3, 128
    wq = np.full((N, K // 8), 0x9ABCDEF0, dtype=np.uint32)
    beta = bf16([-0.375, 0.5, 2.0])
    w = weights(wq, np.zeros((N, K // 64)), np.repeat(beta[:, None], K // 64, 1), N, K, 4)
    y, _ = oracle.qlinear(np.ones((2, K)), w)
    assert np.all(y == np.array([-0.375, 0.5, 2.0]) * K)


def test_constant_code_power_of_two_scale_random_x():
    # q = 11, s = 2^-j, b = 0, random x  ->  y = s * 11 * sum(x)
    rng = np.random.default_rng(7)
    N, K = 6, 512
    wq = np.full((N, K // 8), 11 * 0x11111111, dtype=np.uint32)
    s = np.array([2.0 ** -j for j in range(N)], dtype=np.float32)
    w = weights(wq, np.repeat(bf16(s)[:, None], K // 64, 1), np.zeros((N, K // 64)), N, K, 4)
    x = rng.standard_normal((3, K))
    y, _ = oracle.qlinear(x, w)
    expect = x.sum(axis=1)[:, None] * (11 * s.astype(np.float64))[None, :]
    np.testing.assert_allclose(y, expect, rtol=1e-12, atol=1e-12)


def test_8bit_constant_code():
    N, K = 2, 128
    wq = np.full((N, K // 4), 0xFFFFFFFF, dtype=np.uint32)
    w = weights(wq, np.full((N, K // 64), ONE), np.zeros((N, K // 64)), N, K, 8)
    y, _ = oracle.qlinear(np.ones((1, K)), w)
    assert np.all(y == 255 * K)


def test_hand_case_4x64x8():
    # q[n][k] = (n + k) mod 16 -> every row holds each code 4 times, sum 480;
    # x[m][k] = m + 1, s_n = 2^-n, b_n = -n/8 (all exact in bf16):
    # y[m][n] = (m + 1) * (480 * 2^-n - 64 * n / 8) = (m + 1) * (480 * 2^-n - 8 n)
    M, K, N = 4, 64, 8
    q = np.array([[(n + k) % 16 for k in range(K)] for n in range(N)])
    s = bf16([2.0 ** -n for n in range(N)])[:, None]
    b = bf16([-n / 8 for n in range(N)])[:, None]
    w = weights(synth.pack_codes(q, 4), s, b, N, K, 4)
    x = np.array([[m + 1] * K for m in range(M)], dtype=np.float64)
    y, _ = oracle.qlinear(x, w)
    expect = np.array([[(m + 1) * (480 * 2.0 ** -n - 8 * n) for n in range(N)] for m in range(M)])
    assert np.array_equal(y, expect)


def test_one_hot_rows_reveal_codes_scales_and_biases():
    # x = e_k picks column k of W: y[k][n] = s_n * ((n + k) mod 16) + b_n
    K, N = 128, 16
    q = np.array([[(n + k) % 16 for k in range(K)] for n in range(N)])
    s = np.array([[0.25, 2.0]] * N, dtype=np.float32)           # group 0, group 1
    b = np.array([[-1.0 - n / 4, 3.0] for n in range(N)], dtype=np.float32)
    w = weights(synth.pack_codes(q, 4), bf16(s), bf16(b), N, K, 4)
    y, _ = oracle.qlinear(np.eye(K), w)
    expect = np.array([[s[n, k // 64] * ((n + k) % 16) + b[n, k // 64] for n in range(N)]
                       for k in range(K)])
    assert np.array_equal(y, expect)


# ---------------------------------------------------------------- invariants

def _random_case(seed, M=3, K=256, N=24, bits=4):
    rng = np.random.default_rng(seed)
    w = synth.quant_weights(rng, N, K, bits)
    x = oracle.bf16_to_f64(synth.activations(rng, M, K))
    return x, w


@pytest.mark.parametrize("bits", [4, 8])
def test_joint_group_permutation_leaves_y(bits):
    x, w = _random_case(3, bits=bits)
    K = w["K"]
    G = K // 64
    per = 32 // bits
    perm = np.random.default_rng(4).permutation(G)
    words_per_group = 64 // per
    wq = w["wq"].reshape(w["N"], G, words_per_group)[:, perm].reshape(w["N"], -1)
    w2 = dict(w, wq=wq, scales=w["scales"][:, perm], biases=w["biases"][:, perm])
    x2 = x.reshape(x.shape[0], G, 64)[:, perm].reshape(x.shape[0], K)
    y1, a1 = oracle.qlinear(x, w)
    y2, a2 = oracle.qlinear(x2, w2)
    np.testing.assert_allclose(y2, y1, rtol=1e-12, atol=1e-12 * np.abs(a1).max())


def test_row_permutation_permutes_y():
    x, w = _random_case(5)
    perm = np.random.default_rng(6).permutation(w["N"])
    w2 = dict(w, wq=w["wq"][perm], scales=w["scales"][perm], biases=w["biases"][perm])
    y1, _ = oracle.qlinear(x, w)
    y2, _ = oracle.qlinear(x, w2)
    assert np.array_equal(y2, y1[:, perm])


def test_rows_of_x_are_independent_and_linear():
    x, w = _random_case(8, M=4)
    y, _ = oracle.qlinear(x, w)
    for m in range(4):
        ym, _ = oracle.qlinear(x[m:m + 1], w)
        assert np.array_equal(ym[0], y[m])
    y2, _ = oracle.qlinear(2.0 * x, w)
    assert np.array_equal(y2, 2.0 * y)


def test_dequant_against_explicit_affine_values():
    # scale 0.5, bias -4 on codes 0..15 gives -4, -3.5, ..., 3.5
    wq = np.array([[0x76543210, 0xFEDCBA98] * 4], dtype=np.uint32)
    w = weights(wq, [[bf16(0.5)]], [[bf16(-4.0)]], 1, 64, 4)
    d = oracle.dequant(w)
    assert d[0, :16].tolist() == [-4 + 0.5 * i for i in range(16)]


# ---------------------------------------------------------------- rmsnorm

def test_rmsnorm_constant_row():
    K = 64
    g = np.linspace(0.5, 1.5, K)
    for c in (-3.0, 0.25, 7.0):
        xn = oracle.rmsnorm(np.full((1, K), c), g, 0.0)
        np.testing.assert_allclose(xn[0], math.copysign(1.0, c) * g, rtol=1e-15)
        eps = 1e-2
        xn = oracle.rmsnorm(np.full((1, K), c), g, eps)
        np.testing.assert_allclose(xn[0], c / math.sqrt(c * c + eps) * g, rtol=1e-15)


def test_rmsnorm_three_four():
    # mean of squares of (3, 4) is 12.5
    xn = oracle.rmsnorm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.0)
    np.testing.assert_allclose(xn[0], [3 / math.sqrt(12.5), 8 / math.sqrt(12.5)], rtol=1e-15)


def test_rmsnorm_scale_invariant_without_eps():
    x = np.random.default_rng(1).standard_normal((2, 96))
    g = np.ones(96)
    np.testing.assert_allclose(oracle.rmsnorm(5.0 * x, g, 0.0), oracle.rmsnorm(x, g, 0.0), rtol=1e-14)


# ---------------------------------------------------------------- swiglu

def test_swiglu_closed_forms():
    ln3 = math.log(3.0)
    g = np.array([0.0, ln3, -ln3, 1000.0, -1000.0, 2.0])
    u = np.array([5.0, 2.0, 2.0, 3.0, 3.0, -1.0])
    h = oracle.swiglu(g, u)
    # sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4
    np.testing.assert_allclose(h[:3], [0.0, 2 * 0.75 * ln3, -2 * 0.25 * ln3], rtol=1e-15, atol=0)
    assert h[3] == 3000.0
    assert h[4] == 0.0 or abs(h[4]) < 1e-300
    np.testing.assert_allclose(h[5], -2.0 / (1.0 + math.exp(-2.0)), rtol=1e-15)


# ---------------------------------------------------------------- routing

def test_topk_matches_sorted_with_ties():
    rng = np.random.default_rng(11)
    # small integers force many exact ties
    logits = rng.integers(-3, 4, size=(6, 128)).astype(np.float32)
    idx, w = oracle.topk_softmax(logits, 8)
    for m in range(6):
        order = sorted(range(128), key=lambda e: (-float(logits[m, e]), e))[:8]
        assert idx[m].tolist() == order
        np.testing.assert_allclose(w[m].sum(), 1.0, rtol=1e-15)
        assert np.all(np.diff(w[m]) <= 0)


def test_topk_softmax_closed_forms():
    logits = np.full((1, 16), -5.0, dtype=np.float32)
    logits[0, 3] = 1.0
    logits[0, 9] = 1.0 - math.log(2.0)
    idx, w = oracle.topk_softmax(logits, 2)
    assert idx.tolist() == [[3, 9]]
    np.testing.assert_allclose(w[0], [2 / 3, 1 / 3], rtol=1e-7)
    idx, w = oracle.topk_softmax(np.zeros((1, 128), np.float32), 8)
    assert idx.tolist() == [list(range(8))]
    np.testing.assert_allclose(w, np.full((1, 8), 1 / 8), rtol=1e-15)


# ---------------------------------------------------------------- moe / chain

def _tiny_moe(seed, identical=False, E=6, H=128, I=64, M=3, top_k=2):
    rng = np.random.default_rng(seed)
    x = oracle.bf16_to_f64(synth.activations(rng, M, H))
    logits = synth.router_logits(rng, M, E)
    mats = {}
    for name, (n, k) in {"gate": (I, H), "up": (I, H), "down": (H, I)}.items():
        w = synth.quant_weights(rng, n, k, 4, batch=E)
        if identical:
            for key in ("wq", "scales", "biases"):
                w[key] = np.repeat(w[key][:1], E, axis=0)
        mats[name] = w
    return x, logits, mats, top_k


def test_moe_with_identical_experts_is_the_dense_mlp():
    x, logits, mats, top_k = _tiny_moe(21, identical=True)
    out = oracle.moe(x, logits, mats["gate"], mats["up"], mats["down"], top_k)
    gu = oracle.gateup(x, oracle.expert(mats["gate"], 0), oracle.expert(mats["up"], 0))
    dense, _ = oracle.qlinear(gu["h"], oracle.expert(mats["down"], 0))
    np.testing.assert_allclose(out["y"], dense, rtol=1e-12, atol=1e-12 * np.abs(dense).max())


def test_moe_top1_is_the_selected_expert():
    x, logits, mats, _ = _tiny_moe(22)
    out = oracle.moe(x, logits, mats["gate"], mats["up"], mats["down"], 1)
    for m in range(x.shape[0]):
        e = int(np.argmax(logits[m]))
        assert out["idx"][m, 0] == e and out["w"][m, 0] == 1.0
        gu = oracle.gateup(x[m:m + 1], oracle.expert(mats["gate"], e), oracle.expert(mats["up"], e))
        d, _ = oracle.qlinear(gu["h"], oracle.expert(mats["down"], e))
        assert np.array_equal(out["y"][m], d[0])


def _tiny_decoder(seed):
    return synth.decoder(seed=seed, n_layers=2, d_model=128, d_ff=192, n_q_heads=2,
                         n_kv_heads=1, head_dim=64, vocab=320, M=2)


def _oracle_layers(cfg):
    layers = []
    for L in cfg["layers"]:
        layers.append({k: (oracle.bf16_to_f64(v) if k.endswith("norm") else v) for k, v in L.items()})
    return layers


def test_decode_step_with_silent_o_and_down_is_the_readout_of_the_input():
    cfg = _tiny_decoder(31)
    for L in cfg["layers"]:
        for name in ("o", "down"):
            L[name]["scales"][:] = 0
            L[name]["biases"][:] = 0
    x = oracle.bf16_to_f64(cfg["x"])
    fn = oracle.bf16_to_f64(cfg["final_norm"])
    out = oracle.decode_step(x, _oracle_layers(cfg), fn, cfg["readout"], cfg["dims"]["q_dim"])
    direct, _ = oracle.qlinear(oracle.rmsnorm(x, fn, 1e-6), cfg["readout"])
    assert np.array_equal(out["logits"], direct)


def test_decode_step_ignores_k_and_v_rows():
    cfg = _tiny_decoder(32)
    x = oracle.bf16_to_f64(cfg["x"])
    fn = oracle.bf16_to_f64(cfg["final_norm"])
    q_dim = cfg["dims"]["q_dim"]
    a = oracle.decode_step(x, _oracle_layers(cfg), fn, cfg["readout"], q_dim)
    for L in cfg["layers"]:
        L["qkv"]["wq"][q_dim:] ^= np.uint32(0x5A5A5A5A)
        L["qkv"]["scales"][q_dim:] = bf16(0.75)
    b = oracle.decode_step(x, _oracle_layers(cfg), fn, cfg["readout"], q_dim)
    assert np.array_equal(a["logits"], b["logits"])
    assert not np.array_equal(a["stages"][0]["qkv"][:, q_dim:], b["stages"][0]["qkv"][:, q_dim:])


# ---------------------------------------------------------------- compositions: bias-only closed forms
#
# With every scale 0 a projection's output is bias * sum(input), the same in every
# column, and with eps = 0 the RMSNorm of a constant row c is sign(c) * gamma exactly.
# Constant rows therefore stay constant through a whole layer, and each composition
# step has a closed form in which swapping two operands (gate and up, the two norms,
# h and h1, a routing weight and its expert) changes the value.

def _silu(v):
    return v / (1.0 + math.exp(-v))


def _bias_only(rng, N, K, beta, bits=4, batch=None):
    """Weights with random codes, zero scales and the constant bias beta (exact in bf16)."""
    w = synth.quant_weights(rng, N, K, bits, batch=batch)
    w["scales"][:] = 0
    w["biases"][:] = bf16(beta)
    return w


def test_gateup_order_and_norm_closed_form():
    # x = 2 (constant), gamma = 0.5, eps = 0: xn = 0.5 everywhere, sum(xn) = K / 2.
    # gate bias 1/32, up bias -1/16 (K = 128): g = 2, u = -4, h = silu(2) * -4.
    rng = np.random.default_rng(41)
    K, N = 128, 24
    gate = _bias_only(rng, N, K, 1 / 32)
    up = _bias_only(rng, N, K, -1 / 16)
    x = np.full((2, K), 2.0)
    out = oracle.gateup(x, gate, up, gamma=np.full(K, 0.5), eps=0.0)
    assert np.array_equal(out["xn"], np.full((2, K), 0.5))
    assert np.array_equal(out["g"], np.full((2, N), 2.0))
    assert np.array_equal(out["u"], np.full((2, N), -4.0))
    np.testing.assert_allclose(out["h"], np.full((2, N), -4.0 * _silu(2.0)), rtol=1e-15, atol=0)
    # the swapped order, silu(u) * g, is a different number
    assert abs(_silu(-4.0) * 2.0 - (-4.0 * _silu(2.0))) > 1.0


def _bias_only_decoder(betas, gammas, n_layers=1, D=128, F=192, q_heads=2, kv_heads=1, hd=64, V=40):
    rng = np.random.default_rng(43)
    Q, KV = q_heads * hd, kv_heads * hd
    layers = []
    for _ in range(n_layers):
        layers.append({"attn_norm": np.full(D, gammas["attn"]), "mlp_norm": np.full(D, gammas["mlp"]),
                       "qkv": _bias_only(rng, Q + 2 * KV, D, betas["qkv"]),
                       "o": _bias_only(rng, D, Q, betas["o"]),
                       "gate": _bias_only(rng, F, D, betas["gate"]),
                       "up": _bias_only(rng, F, D, betas["up"]),
                       "down": _bias_only(rng, D, F, betas["down"])})
    readout = _bias_only(rng, V, D, betas["readout"])
    return layers, np.full(D, gammas["final"]), readout, Q


def test_decode_step_mlp_branch_closed_form():
    # D = 128, Q = 128, F = 192, input row h = 1, eps = 0.
    #   attention norm (gamma 0.5): xn = 0.5, sum = 64; qkv = 64/64 = 1 (every column)
    #   o = -1/16 * Q * 1 = -8;  h1 = 1 - 8 = -7
    #   MLP norm (gamma 0.25) of the negative row -7: -0.25, sum S = -32
    #   g = S/32 = -1, u = -S/16 = 2, a = silu(-1) * 2 (every column)
    #   d = F/64 * a = 3 a;  h2 = h1 + d = -7 + 6 silu(-1)
    #   readout (final gamma 2, bias 1/256): rmsnorm(h2) = -2, sum = -256 -> logits = -1
    # Taking the attention norm for the MLP (S = -64), h instead of h1 as the MLP input
    # (S = +32), h instead of h1 in the residual (h2 = 1 + d) or gate and up swapped
    # each gives another h2.
    betas = {"qkv": 1 / 64, "o": -1 / 16, "gate": 1 / 32, "up": -1 / 16, "down": 1 / 64, "readout": 1 / 256}
    gammas = {"attn": 0.5, "mlp": 0.25, "final": 2.0}
    layers, fn, readout, Q = _bias_only_decoder(betas, gammas)
    x = np.ones((2, 128))
    out = oracle.decode_step(x, layers, fn, readout, Q, eps=0.0)
    st = out["stages"][0]
    assert np.array_equal(st["qkv"], np.ones((2, Q + 128)))
    assert np.array_equal(st["h1"], np.full((2, 128), -7.0))
    a = 2.0 * _silu(-1.0)
    np.testing.assert_allclose(st["gu"]["h"], np.full((2, 192), a), rtol=1e-15, atol=0)
    h2 = -7.0 + 3.0 * a
    np.testing.assert_allclose(st["h2"], np.full((2, 128), h2), rtol=1e-15, atol=0)
    np.testing.assert_allclose(out["logits"], np.full((2, 40), -1.0), rtol=1e-14, atol=0)
    wrong = {"attention norm in the MLP": -7.0 + 3.0 * 4.0 * _silu(-2.0),  # S = -64: g = -2, u = 4
             "h as MLP input": -7.0 + 3.0 * (-2.0) * _silu(1.0),           # S = +32: g = 1, u = -2
             "h in the residual": 1.0 + 3.0 * a,
             "gate and up swapped": -7.0 + 3.0 * (-1.0) * _silu(2.0)}
    for name, v in wrong.items():
        assert abs(v - h2) > 0.1, name


def test_decode_step_two_layers_chain_the_residual():
    # Layer 1 starts from layer 0's h2 < 0: its attention norm gives -0.5, qkv = -1,
    # o = +8, h1' = h2 + 8 > -7; the MLP norm of h1' is -0.25 only while h1' < 0,
    # which holds (h2 + 8 = 1 + 6 silu(-1) < 0), so a is unchanged and h2' = h1' + 3 a.
    betas = {"qkv": 1 / 64, "o": -1 / 16, "gate": 1 / 32, "up": -1 / 16, "down": 1 / 64, "readout": 1 / 256}
    gammas = {"attn": 0.5, "mlp": 0.25, "final": 2.0}
    layers, fn, readout, Q = _bias_only_decoder(betas, gammas, n_layers=2)
    out = oracle.decode_step(np.ones((1, 128)), layers, fn, readout, Q, eps=0.0)
    a = 2.0 * _silu(-1.0)
    h2 = -7.0 + 3.0 * a
    h1b = h2 + 8.0
    assert h1b < 0
    np.testing.assert_allclose(out["stages"][1]["h1"], np.full((1, 128), h1b), rtol=1e-13, atol=0)
    np.testing.assert_allclose(out["h"], np.full((1, 128), h1b + 3.0 * a), rtol=1e-13, atol=0)


def test_moe_pairs_each_weight_with_its_expert():
    # H = 128, I = 64, x = 1. Bias-only experts: o(e) = b_d * I * silu(b_g H) * b_u H.
    #   expert 0: b_g = 1/64, b_u = 1/128, b_d = 1/32  -> o = 2 silu(2)
    #   expert 1: b_g = -1/128, b_u = 1/32, b_d = 1/64 -> o = 4 silu(-1)
    #   experts 2, 3 (never chosen): o = 4 silu(1), 4 silu(3)
    # Row 0 prefers expert 1 (logit 1 against 1 - ln 2), row 1 expert 0; weights 2/3, 1/3.
    H, I, E = 128, 64, 4
    rng = np.random.default_rng(47)
    bg = [1 / 64, -1 / 128, 1 / 128, 3 / 128]
    bu = [1 / 128, 1 / 32, 1 / 64, 1 / 64]
    bd = [1 / 32, 1 / 64, 1 / 32, 1 / 32]
    mats = {}
    for name, (n, k, beta) in {"gate": (I, H, bg), "up": (I, H, bu), "down": (H, I, bd)}.items():
        w = synth.quant_weights(rng, n, k, 4, batch=E)
        w["scales"][:] = 0
        for e in range(E):
            w["biases"][e] = bf16(beta[e])
        mats[name] = w
    o = [bd[e] * I * _silu(bg[e] * H) * bu[e] * H for e in range(E)]
    np.testing.assert_allclose(o, [2 * _silu(2.0), 4 * _silu(-1.0), 4 * _silu(1.0), 4 * _silu(3.0)],
                               rtol=1e-15)
    logits = np.full((2, E), -4.0, dtype=np.float32)
    logits[0, 1], logits[0, 0] = 1.0, 1.0 - math.log(2.0)
    logits[1, 0], logits[1, 1] = 1.0, 1.0 - math.log(2.0)
    out = oracle.moe(np.ones((2, H)), logits, mats["gate"], mats["up"], mats["down"], 2)
    assert out["idx"].tolist() == [[1, 0], [0, 1]]
    np.testing.assert_allclose(out["w"], [[2 / 3, 1 / 3]] * 2, rtol=1e-7)
    for m, (e0, e1) in enumerate([(1, 0), (0, 1)]):
        w0, w1 = out["w"][m]
        np.testing.assert_allclose(out["y"][m], np.full(H, w0 * o[e0] + w1 * o[e1]), rtol=1e-14, atol=0)
        assert abs((w0 * o[e1] + w1 * o[e0]) - (w0 * o[e0] + w1 * o[e1])) > 0.1


# ------------------------------------------------------------------ input Hadamard transform

def _signs_to_pm1(signs, K):
    bits = np.unpackbits(np.asarray(signs, np.uint8), bitorder="little")[:K]
    return 1.0 - 2.0 * bits.astype(np.float64)


@pytest.mark.parametrize("block", [64, 16, 256])
def test_rht_matches_the_library_hadamard_matrix(block):
    # scipy's Sylvester Hadamard matrix, the sign vector unpacked with numpy: the
    # oracle's butterflies must give exactly H (d * x) / sqrt(block) per block
    from scipy.linalg import hadamard
    rng = np.random.default_rng(500 + block)
    M, K = 3, 512
    x = rng.standard_normal((M, K))
    signs = synth.rht_signs(rng, K)
    d = _signs_to_pm1(signs, K)
    H = hadamard(block).astype(np.float64) / math.sqrt(block)
    expect = np.concatenate([(H @ (d[k0:k0 + block] * x[:, k0:k0 + block]).T).T for k0 in range(0, K, block)], axis=1)
    np.testing.assert_allclose(oracle.rht(x, signs, block), expect, rtol=0, atol=1e-12)


def test_rht_is_orthonormal_and_undone_by_its_transpose():
    rng = np.random.default_rng(510)
    M, K = 4, 1024
    x = rng.standard_normal((M, K))
    signs = synth.rht_signs(rng, K)
    xr = oracle.rht(x, signs)
    np.testing.assert_allclose(np.linalg.norm(xr, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    # H is symmetric and orthonormal: applying it again without signs, then the signs, gives x back
    back = oracle.rht(xr, np.zeros_like(signs)) * _signs_to_pm1(signs, K)
    np.testing.assert_allclose(back, x, rtol=0, atol=1e-12)


def test_rht_with_rotated_weights_leaves_the_projection():
    # weights quantised in the rotated basis: W_r = W (D H / 8) per group; then
    # W_r . rht(x) = W . x (the rotation the transform exists to apply)
    rng = np.random.default_rng(520)
    M, K, N = 2, 256, 40
    x = rng.standard_normal((M, K))
    W = rng.standard_normal((N, K))
    signs = synth.rht_signs(rng, K)
    W_r = oracle.rht(W, signs)  # each row of W rotated the same way
    np.testing.assert_allclose(W_r @ oracle.rht(x, signs).T, W @ x.T, rtol=1e-12, atol=1e-10)


def test_rht_single_column_block_flips_signs_only():
    rng = np.random.default_rng(530)
    x = rng.standard_normal((2, 64))
    signs = synth.rht_signs(rng, 64)
    np.testing.assert_array_equal(oracle.rht(x, signs, block=1), x * _signs_to_pm1(signs, 64))


def test_rht_rejects_a_block_that_is_not_a_power_of_two():
    with pytest.raises(ValueError):
        oracle.rht(np.zeros((1, 96)), np.zeros(12, np.uint8), block=48)


# ---------------------------------------------------------------- NVFP4 weight code

# FP4 E2M1 magnitudes as tabulated in the OCP Microscaling Formats specification
# (v1.0, element data types): codes 0..7 in order; codes 8..15 are their negatives.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _torch_e4m3(byte_values):
    torch = pytest.importorskip("torch")
    b = torch.from_numpy(np.ascontiguousarray(byte_values, dtype=np.uint8))
    return b.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_matches_the_library_float8_for_every_byte():
    lib = _torch_e4m3(np.arange(256))
    mine = np.array([oracle.e4m3(c) for c in range(256)])
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(lib))
    assert np.isnan(mine).sum() == 2  # S.1111.111 only; no infinities
    ok = ~np.isnan(lib)
    np.testing.assert_array_equal(mine[ok], lib[ok])
    np.testing.assert_array_equal(np.signbit(mine[ok]), np.signbit(lib[ok]))


def test_e2m1_is_the_published_fp4_grid():
    vals = [oracle.e2m1(c) for c in range(16)]
    assert vals[:8] == E2M1_MAGNITUDES
    assert [-v for v in vals[8:]] == E2M1_MAGNITUDES
    assert math.copysign(1.0, vals[8]) == -1.0  # code 8 is -0


def _nvfp4(codes, scales, gscale, N, K):
    return {"code": "nvfp4", "codes": np.asarray(codes, np.uint8), "scales": np.asarray(scales, np.uint8),
            "gscale": np.float32(gscale), "N": N, "K": K}


def test_nvfp4_dequant_low_nibble_first_and_16_column_blocks():
    N, K = 2, 64
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.zeros((N, K // 16), np.uint8)
    codes[1, 5] = 0x21   # columns 10 (low nibble: 0.5) and 11 (high nibble: 1.0)
    codes[1, 8] = 0xF3   # columns 16 (1.5) and 17 (-6)
    codes[0, 31] = 0x70  # columns 62 (0) and 63 (6)
    scales[1, 0] = 0x38  # 1.0 for columns 0..15
    scales[1, 1] = 0x40  # 2.0 for columns 16..31
    scales[0, 3] = 0x01  # 2^-9 for columns 48..63
    w = oracle.dequant(_nvfp4(codes, scales, 0.25, N, K))
    expect = np.zeros((N, K))
    expect[1, 10], expect[1, 11] = 0.25 * 0.5, 0.25 * 1.0
    expect[1, 16], expect[1, 17] = 0.25 * 2.0 * 1.5, -0.25 * 2.0 * 6.0
    expect[0, 63] = 0.25 * 2.0 ** -9 * 6.0
    np.testing.assert_array_equal(w, expect)


def test_nvfp4_projection_equals_a_matmul_of_an_independent_dequantisation():
    rng = np.random.default_rng(77)
    N, K, M = 40, 192, 3
    w = synth.nvfp4_weights(rng, N, K)
    x = rng.standard_normal((M, K))
    # dequantised separately: nibble split by numpy, the published E2M1 grid, the
    # library's E4M3 conversion, scales repeated over their 16 columns
    lo, hi = w["codes"] & 15, w["codes"] >> 4
    q = np.stack([lo, hi], axis=-1).reshape(N, K)
    grid = np.array(E2M1_MAGNITUDES + [-v for v in E2M1_MAGNITUDES])
    W = float(w["gscale"]) * np.repeat(_torch_e4m3(w["scales"]), 16, axis=1) * grid[q]
    y, ad = oracle.qlinear(x, w)
    np.testing.assert_allclose(y, x @ W.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ad, np.abs(x) @ np.abs(W).T, rtol=1e-12, atol=1e-12)


def test_nvfp4_global_scale_scales_the_projection():
    rng = np.random.default_rng(78)
    w = synth.nvfp4_weights(rng, 16, 128)
    x = rng.standard_normal((2, 128))
    y1, _ = oracle.qlinear(x, w)
    y2, _ = oracle.qlinear(x, dict(w, gscale=np.float32(w["gscale"]) * np.float32(8.0)))
    np.testing.assert_array_equal(y2, 8.0 * y1)  # a power of two changes no rounding


def test_decode_step_readout_row_subset_nvfp4():
    # the readout restricted to a set of vocabulary rows equals those rows of the full one
    cfg = synth.decoder(seed=79, n_layers=1, d_model=128, d_ff=192, n_q_heads=2, n_kv_heads=1, head_dim=64,
                        vocab=300, M=2, code="nvfp4")
    layers = [{k: (oracle.bf16_to_f64(v) if k.endswith("norm") else v) for k, v in L.items()} for L in cfg["layers"]]
    x = oracle.bf16_to_f64(cfg["x"])
    fn = oracle.bf16_to_f64(cfg["final_norm"])
    full = oracle.decode_step(x, layers, fn, cfg["readout"], cfg["dims"]["q_dim"])
    rows = np.array([299, 0, 17, 150])
    sub = oracle.decode_step(x, layers, fn, cfg["readout"], cfg["dims"]["q_dim"], readout_rows=rows)
    np.testing.assert_array_equal(sub["logits"], full["logits"][:, rows])
