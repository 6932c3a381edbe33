"""Benchmark of the quantised decode projection on GB300.

Default workload (one JSON line): the fused RMSNorm + gate/up SwiGLU projection,
4-bit group-64 weights, K=1024, N=2x3072; one step is one M=1 call followed by
one M=8 call, each on its own copy of the weights from a rotation of copies
whose total is more than four times the L2 cache, so every call streams its
weights from HBM. Steps are captured once into a CUDA graph and replayed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tfq|reference]
                  [--workload gateup|proj|wide|step|moe4|moe8|all]

value      effective weight GB/s: algorithmic weight bytes (codes + scales +
           biases) of all calls / device time of the timed region.
e2e        the same metric with the per-step activations copied in from pinned
           host memory and the outputs copied back inside the timed region.
roofline   the dominant kernel's bytes per launch / its mean launch time against
           the measured HBM copy bandwidth.
cpu_baseline  the fp64 oracle on a bounded sample, on this host's cores.

Under torchrun (N > 1) every rank runs an independent replica of the workload
(replicas: the projection has no exchange step); the timed region is bracketed by
barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective weight GB/s & % of HBM peak per quantized projection at M=1 and M=8"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "skinny_gemm_bit_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(kernel_key)
        if rec and rec.get("source_hash") == kernel_source_hash():
            return float(rec["bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


# ----------------------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("TFQ_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def max_over_ranks(value: float, pg, device) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def barrier(pg):
    if pg is not None:
        pg.barrier()


# ----------------------------------------------------------------------------- workloads

class Workload:
    """A sequence of calls per step over rotating weight copies."""

    name = ""
    kernel_key = ""

    def __init__(self, T, torch, copies_bytes_min: int):
        self.T = T
        self.torch = torch

    def weight_bytes_per_step(self) -> int:
        raise NotImplementedError

    def step(self, i: int, flags: int):
        raise NotImplementedError

    def step_e2e(self, i: int, flags: int):
        raise NotImplementedError


def _dev_bf16(torch, u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).cuda().view(torch.bfloat16)


def _rotations(per_copy_bytes: int, l2_bytes: int) -> int:
    return max(2, int(np.ceil(4 * l2_bytes / per_copy_bytes)) + 1)


def _clone_qweight(T, qw):
    buf = qw.buf.clone()
    desc = type(qw.desc).from_buffer_copy(qw.desc)
    desc.data = buf.data_ptr()
    return T.QWeight(buf, desc)


class GateUp(Workload):
    """Fused RMSNorm + gate/up SwiGLU, K=1024, N=2x3072; one M=1 and one M=8 call per step."""

    kernel_key = "qproj_b4_dual_k1024_n3072"

    def __init__(self, T, torch, l2_bytes, K=1024, N=3072):
        from skinny_gemm_bit_gb300 import synth
        self.T, self.torch = T, torch
        cfg = synth.fused_gateup(seed=1, M=8, K=K, N=N)
        self.K, self.N = K, N
        g = T.tf_qlinear_pack(cfg["gate"]["wq"], cfg["gate"]["scales"], cfg["gate"]["biases"], 4)
        u = T.tf_qlinear_pack(cfg["up"]["wq"], cfg["up"]["scales"], cfg["up"]["biases"], 4)
        self.per_call = g.weight_bytes() + u.weight_bytes()
        n = _rotations(g.buf.numel() + u.buf.numel(), l2_bytes)
        self.copies = [(g, u)] + [(_clone_qweight(T, g), _clone_qweight(T, u)) for _ in range(n - 1)]
        self.gamma = _dev_bf16(torch, cfg["gamma"])
        self.eps = cfg["eps"]
        self.x8 = _dev_bf16(torch, cfg["x"])
        self.x1 = self.x8[:1].clone()
        self.h1 = torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
        self.h8 = torch.empty((8, N), dtype=torch.bfloat16, device="cuda")
        self.ws = T.workspace(T.tf_qmlp_gateup_workspace_bytes(g, u, 8))
        # host side of the end-to-end variant
        self.x1_h = self.x1.cpu().pin_memory()
        self.x8_h = self.x8.cpu().pin_memory()
        self.h1_h = torch.empty_like(self.h1, device="cpu").pin_memory()
        self.h8_h = torch.empty_like(self.h8, device="cpu").pin_memory()
        self.n_copies = n
        self.launches_per_step = 2
        self.desc = (f"fused RMSNorm + gate/up SwiGLU projection, 4-bit group-64, K={K}, N=2x{N}; "
                     f"one M=1 and one M=8 call per step")

    def weight_bytes_per_step(self):
        return 2 * self.per_call

    def _calls(self, i, flags):
        g, u = self.copies[(2 * i) % self.n_copies]
        self.T.tf_qmlp_gateup_run(g, u, self.x1, self.gamma, self.eps, out=self.h1, ws=self.ws, flags=flags)
        g, u = self.copies[(2 * i + 1) % self.n_copies]
        self.T.tf_qmlp_gateup_run(g, u, self.x8, self.gamma, self.eps, out=self.h8, ws=self.ws, flags=flags)

    def step(self, i, flags):
        self._calls(i, flags)

    def step_e2e(self, i, flags):
        self.x1.copy_(self.x1_h, non_blocking=True)
        self.x8.copy_(self.x8_h, non_blocking=True)
        self._calls(i, 0)
        self.h1_h.copy_(self.h1, non_blocking=True)
        self.h8_h.copy_(self.h8, non_blocking=True)

    def io_bytes(self):
        return (self.x1.numel() + self.x8.numel()) * 2, (self.h1.numel() + self.h8.numel()) * 2

    def per_m(self, flags, reps=200):
        """Mean device time per call for M=1 and M=8 separately (graph-replayed)."""
        out = {}
        for M, x, h in ((1, self.x1, self.h1), (8, self.x8, self.h8)):
            def one(i):
                g, u = self.copies[i % self.n_copies]
                self.T.tf_qmlp_gateup_run(g, u, x, self.gamma, self.eps, out=h, ws=self.ws, flags=flags)
            ms = time_graph(self.torch, one, reps)
            out[M] = ms * 1e3 / reps
        return out

    def oracle_sample(self, seconds: float):
        """Run the fp64 oracle on gate/up rows for about `seconds`; returns (weight bytes, s, desc)."""
        import oracle
        from skinny_gemm_bit_gb300 import synth
        cfg = synth.fused_gateup(seed=1, M=8, K=self.K, N=self.N)
        rows = 256
        sub = lambda w: {"wq": w["wq"][:rows], "scales": w["scales"][:rows], "biases": w["biases"][:rows],  # noqa
                         "N": rows, "K": w["K"], "bits": w["bits"]}
        g, u = sub(cfg["gate"]), sub(cfg["up"])
        x = oracle.bf16_to_f64(cfg["x"])
        gam = oracle.bf16_to_f64(cfg["gamma"])
        done, t0, reps = 0, time.perf_counter(), 0
        while True:
            for M in (1, 8):
                oracle.gateup(x[:M], g, u, gam, cfg["eps"])
                done += 2 * rows * self.K * (4 / 8 + 4 / 64)
            reps += 1
            if time.perf_counter() - t0 >= seconds:
                break
        el = time.perf_counter() - t0
        return done, el, (f"{reps} x (M=1 and M=8 calls of the fused RMSNorm + gate/up oracle on the first "
                          f"{rows} of {self.N} rows of each matrix, K={self.K}), single thread")


def time_graph(torch, fn, n):
    """Capture n calls fn(0..n-1) into a CUDA graph; return device ms of one replay (after 3 warm replays)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(min(n, 3)):
            fn(i)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            fn(i)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b)


# ----------------------------------------------------------------------------- main

def run_tfq(args):
    import torch
    world, rank, local, pg = dist_setup()
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    from skinny_gemm_bit_gb300 import tfq as T

    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024) or 126 * 1024 * 1024
    wl = GateUp(T, torch, l2)
    flags = T.TF_RUN_PDL
    K, W = args.steps, args.warmup

    # capture K timed steps (and W warm-up steps) into graphs
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        wl.step(0, flags)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g_warm, g_timed = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_warm):
        for i in range(W):
            wl.step(i, flags)
    with torch.cuda.graph(g_timed):
        for i in range(K):
            wl.step(W + i, flags)
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e):
        for i in range(K):
            wl.step_e2e(W + i, flags)

    sampler = ClockSampler(local)
    sampler.start()
    g_warm.replay()
    # keep the GPU busy for ~1 s so the clock samples cover a loaded state
    t_end = time.time() + 1.0
    while time.time() < t_end:
        g_timed.replay()
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    g_timed.replay()
    ev1.record()
    torch.cuda.synchronize()
    barrier(pg)
    ms = ev0.elapsed_time(ev1)
    clocks = sampler.stop()
    ms_max = max_over_ranks(ms, pg, f"cuda:{local}")

    # end to end: host buffers in, host buffers out, inside the timed region
    g_e2e.replay()
    torch.cuda.synchronize()
    barrier(pg)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g_e2e.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(pg)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), pg, f"cuda:{local}")

    per_m = wl.per_m(flags)
    per_m_nopdl = wl.per_m(0)

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return
    peak, peak_kind = measured_peaks()
    bytes_step = wl.weight_bytes_per_step()
    value = world * bytes_step * K / (ms_max * 1e-3) / 1e9
    e2e_value = world * bytes_step * K / (ms_e2e * 1e-3) / 1e9
    launch_us = ms_max * 1e3 / (K * wl.launches_per_step)
    achieved = wl.per_call / (launch_us * 1e-6) / 1e9
    cpu = cpu_baseline(wl, args.cpu_seconds)
    h2d, d2h = wl.io_bytes()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms_max / K, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded random 4-bit weights and N(0,1) activations)",
        "config": {"workload": wl.desc, "K": wl.K, "N": 2 * wl.N, "M": [1, 8], "bits": 4, "group": 64,
                   "l2": f"weights rotate over {wl.n_copies} copies ({wl.n_copies * bytes_step / 2 / 1e6:.0f} MB, "
                         f"> 4x L2), every call reads HBM", "graph": "CUDA graph, programmatic dependent launch",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_hbm_measured": round(100 * value / world / peak, 2),
        "pct_of_8tbs_nominal": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "per_m": {str(M): {"us_per_call": round(us, 3), "gbs": round(wl.per_call / (us * 1e-6) / 1e9, 1)}
                  for M, us in per_m.items()},
        "per_m_no_pdl": {str(M): {"us_per_call": round(us, 3), "gbs": round(wl.per_call / (us * 1e-6) / 1e9, 1)}
                         for M, us in per_m_nopdl.items()},
        "m8_over_m1": round(per_m[8] / per_m[1], 3),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": recorded_traffic(wl.kernel_key),
                     "peak_source": peak_kind, "kernel": "qproj_kernel<4, dual>",
                     "bytes_per_launch": wl.per_call, "launch_us": round(launch_us, 3)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": K * wl.launches_per_step,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def cpu_baseline(wl, seconds):
    done, el, desc = wl.oracle_sample(seconds)
    return {"value": round(done / el / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc}


def run_reference(args):
    """The fp64 oracle as the reference arm, on this host's cores, rank 0 only."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    class _Host:
        pass

    wl = GateUp.__new__(GateUp)
    wl.K, wl.N = 1024, 3072
    desc = None
    steps_s = []
    oracle.build()
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        done, el, desc = wl.oracle_sample(args.ref_step_seconds)
        if i >= args.warmup:
            steps_s.append((done, el))
    total_b = sum(d for d, _ in steps_s)
    total_s = sum(e for _, e in steps_s)
    value = total_b / total_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total_s / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded random 4-bit weights and N(0,1) activations)",
        "config": {"workload": "fused RMSNorm + gate/up SwiGLU projection, 4-bit group-64, K=1024, N=2x3072; "
                               "one M=1 and one M=8 call per step", "K": 1024, "N": 6144, "M": [1, 8],
                   "bits": 4, "group": 64},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "kind": "oracle", "cores": 1,
                         "sample": f"each step: {desc}"},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="tfq", choices=["tfq", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-step-seconds", type=float, default=0.2)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_tfq(args)


if __name__ == "__main__":
    main()
