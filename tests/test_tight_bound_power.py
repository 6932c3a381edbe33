"""The tight GPU bounds discriminate: planted mistakes, on the CPU, fall outside them."""
import numpy as np

import oracle
from parity import NORM_TIGHT, PLAIN_TIGHT, TINY
from skinny_gemm_bit_gb300 import synth


def test_a_dropped_group_falls_outside_the_plain_bound():
    # the oracle's result with one 64-column group of every row left out stands in
    # for a kernel that skips a group
    rng = np.random.default_rng(5)
    M, K, N = 4, 1024, 64
    x = oracle.bf16_to_f64(synth.activations(rng, M, K))
    w = synth.quant_weights(rng, N, K, 4)
    ref, ad = oracle.qlinear(x, w)
    x_drop = x.copy()
    x_drop[:, 320:384] = 0.0
    dropped, _ = oracle.qlinear(x_drop, w)
    assert np.mean(np.abs(dropped - ref) > PLAIN_TIGHT * ad + TINY) > 0.9


def test_an_unnormalised_row_falls_outside_the_norm_bound():
    # a kernel that skipped the RMSNorm factor (gamma applied, 1 / rms not) would be
    # off by the row's scale; here rms is about 1, so scale the input to make it 3
    rng = np.random.default_rng(6)
    M, K, N = 2, 1024, 64
    x = 3.0 * oracle.bf16_to_f64(synth.activations(rng, M, K))
    g = oracle.bf16_to_f64(synth.gamma(rng, K))
    w = synth.quant_weights(rng, N, K, 4)
    ref, ad = oracle.qlinear(oracle.rmsnorm(x, g, 1e-6), w)
    wrong, _ = oracle.qlinear(x * g, w)
    assert np.mean(np.abs(wrong - ref) > NORM_TIGHT * ad + TINY) > 0.9


def test_the_tight_bounds_are_tighter_than_the_stated_one():
    assert PLAIN_TIGHT < NORM_TIGHT < 1e-2 / 4
