"""bench.py's host side without a GPU: every workload's oracle sample (the reference
arm and the cpu_baseline leg) runs and reports the bytes it covered."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("name", [w for w in bench.WORKLOADS if w not in ("step", "verify", "readout",
                                                                           "readout_nvfp4")])
def test_every_workload_has_an_oracle_sample(name):
    host = bench._HostOnly(name)
    done, seconds, desc = host.oracle_sample(0.01)
    assert done > 0 and seconds > 0 and "oracle" in desc
    assert host.desc


def test_nvfp4_sample_counts_nvfp4_bytes():
    host = bench._HostOnly("wide_nvfp4")
    done, _, _ = host.oracle_sample(0.01)
    rows, K = 32, 12800
    per_call = rows * K * (0.5 + 1 / 16)
    assert done % per_call == 0 and "NVFP4" in host.desc


def test_reference_arm_names_the_gpu_arms_workloads():
    # both arms print the same config["workload"], so their lines describe one config
    assert bench._HostOnly("step").desc == bench.STEP_DESC
    assert bench._HostOnly("gateup").desc == bench.gateup_desc(1024, 3072)
    for name, (K, N, ms) in {"proj": (1024, 3072, (1,)), "wide": (12800, 2560, (1, 8)),
                             "wide_nvfp4": (12800, 2560, (1, 8))}.items():
        assert bench._HostOnly(name).desc == bench.proj_desc(name, K, N, ms)
    assert bench._HostOnly("moe4").desc == bench.moe_desc(False, 4, 56)
