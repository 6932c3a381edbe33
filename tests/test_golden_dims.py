"""The decoder-step workload against the model dimensions the pages print
(tests/golden/qwen3_0p6b_decoder_dims.txt, with its citation)."""
import os

import numpy as np

from skinny_gemm_bit_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    vals = {}
    with open(os.path.join(HERE, "golden", "qwen3_0p6b_decoder_dims.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


def test_decoder_workload_has_the_printed_dimensions():
    g = _golden()
    cfg = synth.decoder(n_layers=1, M=1)  # one layer is enough to read the shapes
    d = cfg["dims"]
    assert (d["d_model"], d["d_ff"], d["vocab"]) == (g["d_model"], g["d_ff"], g["vocab"])
    assert synth.decoder.__defaults__[1] == g["n_layers"]  # n_layers default
    L = cfg["layers"][0]
    assert L["gate"]["N"] == L["up"]["N"] == g["d_ff"] and L["down"]["K"] == g["d_ff"]
    assert cfg["readout"]["N"] == g["vocab"] and cfg["readout"]["K"] == g["d_model"]
    # the step's weight bytes at 0.5625 B a weight (4-bit codes, a bf16 scale and bias per 64)
    per_layer = sum(L[k]["N"] * L[k]["K"] for k in ("qkv", "o", "gate", "up", "down"))
    total = (g["n_layers"] * per_layer + g["vocab"] * g["d_model"]) * 0.5625
    assert total == 335241216
    assert np.isclose(per_layer, 15.73e6, rtol=1e-3)
