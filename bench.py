"""Benchmark of the quantised decode projection on GB300.

Default workload (one JSON line): the per-token weight stream of a 28-layer dense
decoder (d_model 1024, d_ff 3072, 16 q / 8 kv heads of 128, tied readout
151,936 x 1024; 4-bit group-64 weights, 335 MB per step): one step is one M=1
decoder step followed by one M=8 decoder step. Each step streams more than twice
L2 from HBM, and L2 is flushed before every timed replay. Steps are captured
once into a CUDA graph and replayed; the timed graph is replayed five times and
the median is reported.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tfq|reference]
                  [--workload step|gateup|proj|wide|wide_rht|readout|moe4|moe8|moe_nvfp4|
                              verify|wide_nvfp4|readout_nvfp4]

The other workloads: gateup (the fused RMSNorm + gate/up SwiGLU projection, K=1024,
N=2x3072, one M=1 and one M=8 call; weights rotate over copies whose total is more
than four times L2), proj (one K=1024, N=3072 projection, M=1), wide (K=12800,
N=2560, one M=1 and one M=8 call), wide_rht (the same with the input Hadamard
transform folded into the activation staging), readout (the decoder's RMSNorm + tied readout,
K=1024, N=151936, one M=1 and one M=8 call), step (the whole per-token weight
stream of a 28-layer dense decoder, one M=1 and one M=8 step), moe4 / moe8 / moe_nvfp4
(the MoE layer, M=8, one call; 4-bit, 8-bit or NVFP4 experts), verify (greedy generation of 64 tokens on that decoder
with prompt-lookup drafts verified up to 8 rows a step; host-driven, timed end to
end, against plain one-token decoding), wide_nvfp4 / readout_nvfp4 (the wide and
readout shapes with NVFP4 weights: E2M1 codes, an E4M3 scale per 16 columns).

value      effective weight GB/s: algorithmic weight bytes (codes + scales +
           biases) of all calls / device time of the timed region (median of five
           timed replays, each after an L2 flush).
e2e        the same metric with the per-step activations copied in from pinned
           host memory and the outputs copied back inside the timed region.
roofline   bytes per call / mean call time of the timed region against the
           measured HBM copy bandwidth; a call is one launch of the named kernel
           (four launches for the MoE layer).
cpu_baseline  the fp64 oracle on a bounded sample, on all of this host's cores (threads
           splitting the sample's rows), with the single-thread figure beside it.

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
REPLAYS = 5
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
    """A sequence of calls per step (one per entry of `step_ms`) over rotating weight copies.

    Subclasses set: name, kernel_key, kernel, desc, K, N, bits, per_call (weight bytes of
    one call), n_copies, and implement call(copy, M, flags, x, out) plus the host sample of
    the oracle."""

    step_ms = (1, 8)

    def __init__(self, T, torch):
        self.T, self.torch = T, torch

    # inputs per M: device tensors (used by the timed steps) and pinned host copies
    def _io(self, x8_u16, out_cols):
        torch = self.torch
        self.x = {}
        self.out = {}
        self.x_h = {}
        self.out_h = {}
        for M in sorted(set(self.step_ms)):
            self.x[M] = _dev_bf16(torch, x8_u16[:M])
            self.out[M] = torch.empty((M, out_cols), dtype=torch.bfloat16, device="cuda")
            self.x_h[M] = self.x[M].cpu().pin_memory()
            self.out_h[M] = torch.empty_like(self.out[M], device="cpu").pin_memory()

    @property
    def launches_per_step(self):
        return len(self.step_ms) * self.launches_per_call

    launches_per_call = 1

    def weight_bytes_per_step(self):
        return len(self.step_ms) * self.per_call

    def step(self, i, flags):
        for j, M in enumerate(self.step_ms):
            self.call((len(self.step_ms) * i + j) % self.n_copies, M, flags, self.x[M], self.out[M])

    def step_e2e(self, i, flags):
        for j, M in enumerate(self.step_ms):
            self.x[M].copy_(self.x_h[M], non_blocking=True)
            self.call((len(self.step_ms) * i + j) % self.n_copies, M, 0, self.x[M], self.out[M])
            self.out_h[M].copy_(self.out[M], non_blocking=True)

    def io_bytes(self):
        return (sum(self.x[M].numel() * 2 for M in self.step_ms),
                sum(self.out[M].numel() * 2 for M in self.step_ms))

    def per_m(self, flags, reps=100):
        """Mean device time per call for each M (graph-replayed)."""
        out = {}
        for M in sorted(set(self.step_ms)):
            def one(i, M=M):
                self.call(i % self.n_copies, M, flags, self.x[M], self.out[M])
            ms = time_graph(self.torch, one, reps)
            out[M] = ms * 1e3 / reps
        return out

    def oracle_sample(self, seconds: float, part=(0, 1)):
        """The fp64 oracle on a row subset of one matrix of the workload, M as in a step,
        for about `seconds`; returns (weight bytes covered, seconds, description).
        part = (i, n): only the i-th of n equal slices of those rows (one host thread's share)."""
        import oracle
        w, rows, what = self.sample_matrix()
        r0, r1 = part[0] * rows // part[1], (part[0] + 1) * rows // part[1]
        n = r1 - r0
        if w.get("code") == "nvfp4":
            sub = dict(w, codes=w["codes"][r0:r1], scales=w["scales"][r0:r1], N=n)
            per = n * w["K"] * (4 / 8 + 1 / 16)
        else:
            sub = {"wq": w["wq"][r0:r1], "scales": w["scales"][r0:r1], "biases": w["biases"][r0:r1],
                   "N": n, "K": w["K"], "bits": w["bits"]}
            per = n * w["K"] * (w["bits"] / 8 + 4 / 64)
        x = oracle.bf16_to_f64(self.sample_x)
        signs = getattr(self, "host_signs", None)  # input Hadamard transform, when the workload has one
        done, t0, reps = 0, time.perf_counter(), 0
        while True:
            for M in self.step_ms:
                if n > 0:
                    oracle.qlinear(x[:M] if signs is None else oracle.rht(x[:M], signs), sub)
                done += per
            reps += 1
            if time.perf_counter() - t0 >= seconds:
                break
        el = time.perf_counter() - t0
        ms = " and ".join(f"M={M}" for M in self.step_ms)
        what_oracle = "projection" if signs is None else "input Hadamard transform + projection"
        return done, el, (f"{reps} x ({ms} calls of the {what_oracle} oracle on the first {rows} rows of {what}, "
                          f"K={w['K']})")


def _dev_bf16(torch, u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).cuda().view(torch.bfloat16)


def _rotations(per_copy_bytes: int, l2_bytes: int) -> int:
    return max(2, int(np.ceil(4 * l2_bytes / per_copy_bytes)) + 1)


def _clone_qweight(T, qw):
    buf = qw.buf.clone()
    desc = type(qw.desc).from_buffer_copy(qw.desc)
    desc.data = buf.data_ptr()
    return T.QWeight(buf, desc)


def _pack(T, w):
    if w.get("code") == "nvfp4":
        return T.tf_qlinear_pack_nvfp4(w["codes"], w["scales"], w["gscale"])
    return T.tf_qlinear_pack(w["wq"], w["scales"], w["biases"], w["bits"])


def _weights_word(wl):
    return "NVFP4" if wl.name.endswith("_nvfp4") else f"{wl.bits}-bit"


def _proj_config(kind):
    """Seeded inputs of the single-matrix workloads (also used by the host-only reference arm)."""
    from skinny_gemm_bit_gb300 import synth
    return {"wide": lambda: synth.wide_verify(seed=2, M=8),
            "wide_rht": lambda: synth.wide_verify(seed=2, M=8),
            "readout": lambda: synth.single_projection(seed=3, M=8, K=1024, N=151936),
            "proj": lambda: synth.single_projection(seed=0, M=1),
            "wide_nvfp4": lambda: synth.nvfp4_projection(seed=8, M=8, K=12800, N=2560),
            "readout_nvfp4": lambda: synth.nvfp4_projection(seed=9, M=8, K=1024, N=151936)}[kind]()


# Workload descriptions, shared by both arms so that their lines name the same config
STEP_DESC = ("per-token weight stream of a 28-layer dense decoder, 4-bit group-64: norm+QKV, O, "
             "norm+gate/up+SwiGLU, down per layer, norm+tied readout 151936x1024; one M=1 and one M=8 step")


def gateup_desc(K, N):
    return (f"fused RMSNorm + gate/up SwiGLU projection, 4-bit group-64, K={K}, N=2x{N}; "
            f"one M=1 and one M=8 call per step")


def proj_desc(kind, K, N, step_ms):
    ms = " and ".join(f"M={M}" for M in step_ms)
    what = {"wide": "wide verify 4-bit group-64", "wide_rht": "input Hadamard transform + wide verify 4-bit group-64",
            "readout": "RMSNorm + tied readout 4-bit group-64", "proj": "single 4-bit group-64",
            "wide_nvfp4": "wide verify NVFP4 (E2M1, E4M3 scale per 16)",
            "readout_nvfp4": "RMSNorm + tied readout NVFP4 (E2M1, E4M3 scale per 16)"}[kind]
    return f"{what} projection, K={K}, N={N}; one {ms} call per step"


def moe_desc(nvfp4, bits, distinct):
    codes = "NVFP4 (E2M1, an E4M3 scale per 16, an fp32 scale per expert)" if nvfp4 else f"{bits}-bit group-64"
    return (f"MoE expert projection, M=8, 128 experts, top-8, hidden 2048, intermediate 768, {codes} "
            f"gate/up/down ({distinct} distinct experts read); one call per step")


class GateUp(Workload):
    """Fused RMSNorm + gate/up SwiGLU, K=1024, N=2x3072; one M=1 and one M=8 call per step."""

    name = "gateup"
    kernel_key = "qproj_b4_dual_k1024_n3072"
    kernel = "qstage_kernel<4, dual> (stage kernel, one CTA per row block)"

    def __init__(self, T, torch, l2_bytes, K=1024, N=3072):
        super().__init__(T, torch)
        from skinny_gemm_bit_gb300 import synth
        cfg = synth.fused_gateup(seed=1, M=8, K=K, N=N)
        self.cfg = cfg
        self.K, self.N, self.bits = K, N, 4
        g, u = _pack(T, cfg["gate"]), _pack(T, cfg["up"])
        self.per_call = g.weight_bytes() + u.weight_bytes()
        n = _rotations(g.buf.numel() + u.buf.numel(), l2_bytes)
        self.copies = [(g, u)] + [(_clone_qweight(T, g), _clone_qweight(T, u)) for _ in range(n - 1)]
        self.n_copies = n
        self.gamma = _dev_bf16(torch, cfg["gamma"])
        self.eps = cfg["eps"]
        self._io(cfg["x"], N)
        self.ws = T.workspace(T.tf_qmlp_gateup_workspace_bytes(g, u, 8))
        self.sample_x = cfg["x"]
        self.desc = gateup_desc(K, N)

    def call(self, i, M, flags, x, out):
        g, u = self.copies[i]
        self.T.tf_qmlp_gateup_run(g, u, x, self.gamma, self.eps, out=out, ws=self.ws, flags=flags)

    def oracle_sample(self, seconds: float, part=(0, 1)):
        """The fused RMSNorm + gate/up oracle on the first 256 rows of each matrix (the
        i-th of n slices of them for part = (i, n))."""
        import oracle
        cfg = self.cfg
        total = 256
        r0, r1 = part[0] * total // part[1], (part[0] + 1) * total // part[1]
        rows = r1 - r0
        sub = lambda w: {"wq": w["wq"][r0:r1], "scales": w["scales"][r0:r1], "biases": w["biases"][r0:r1],  # noqa
                         "N": rows, "K": w["K"], "bits": w["bits"]}
        g, u = sub(cfg["gate"]), sub(cfg["up"])
        x = oracle.bf16_to_f64(cfg["x"])
        gam = oracle.bf16_to_f64(cfg["gamma"])
        done, t0, reps = 0, time.perf_counter(), 0
        while True:
            for M in (1, 8):
                if rows > 0:
                    oracle.gateup(x[:M], g, u, gam, cfg["eps"])
                done += 2 * rows * self.K * (4 / 8 + 4 / 64)
            reps += 1
            if time.perf_counter() - t0 >= seconds:
                break
        el = time.perf_counter() - t0
        return done, el, (f"{reps} x (M=1 and M=8 calls of the fused RMSNorm + gate/up oracle on the first "
                          f"{total} of {self.N} rows of each matrix, K={self.K})")


class Proj(Workload):
    """One 4-bit projection per step: K=1024, N=3072, M=1 (single projection); K=12800,
    N=2560 at M=1 and M=8 (wide verify projection); or the decoder's tied readout with
    its RMSNorm, K=1024, N=151936, at M=1 and M=8. The *_nvfp4 kinds are the wide and
    readout shapes with NVFP4 weights."""

    def __init__(self, T, torch, l2_bytes, kind: str):
        super().__init__(T, torch)
        from skinny_gemm_bit_gb300 import synth
        self.gamma, self.eps, self.signs = None, 1e-6, None
        cfg = _proj_config(kind)
        if kind == "wide_nvfp4":
            self.name, self.step_ms = kind, (1, 8)
            self.kernel_key = "qproj_nvfp4_k12800_n2560"
            self.kernel = "qproj_warp_kernel<NVFP4> (warp workers, K split in 5)"
        elif kind == "readout_nvfp4":
            self.name, self.step_ms = kind, (1, 8)
            self.kernel_key, self.kernel = "qproj_nvfp4_k1024_n151936_norm", "qproj_warp_kernel<NVFP4> (warp workers)"
            self.gamma = _dev_bf16(torch, synth.gamma(np.random.default_rng(5), 1024))
        elif kind == "wide_rht":
            self.name, self.step_ms = "wide_rht", (1, 8)
            self.kernel_key = "qproj_b4_k12800_n2560_rht"
            self.kernel = "qproj_warp_kernel<4> (warp workers, K split, input Hadamard transform at staging)"
            self.host_signs = synth.rht_signs(np.random.default_rng(2), 12800)
            self.signs = torch.from_numpy(self.host_signs).cuda()
        elif kind == "wide":
            self.name, self.step_ms = "wide", (1, 8)
            self.kernel_key = "qproj_b4_k12800_n2560"
            self.kernel = "qproj_warp_kernel<4> (warp workers, K split in 5)"
        elif kind == "readout":
            self.name, self.step_ms = "readout", (1, 8)
            self.kernel_key, self.kernel = "qproj_b4_k1024_n151936_norm", "qproj_warp_kernel<4> (warp workers)"
            self.gamma = _dev_bf16(torch, synth.gamma(np.random.default_rng(5), 1024))
        else:
            self.name, self.step_ms = "proj", (1,)
            self.kernel_key, self.kernel = "qproj_b4_k1024_n3072", "qstage_kernel<4> (stage kernel, one CTA per row block)"
        w0 = _pack(T, cfg["w"])
        self.w = cfg["w"]
        self.K, self.N, self.bits = w0.K, w0.N, 4
        self.per_call = w0.weight_bytes()
        n = _rotations(w0.buf.numel(), l2_bytes)
        self.copies = [w0] + [_clone_qweight(T, w0) for _ in range(n - 1)]
        self.n_copies = n
        x8 = cfg["x"] if cfg["x"].shape[0] == 8 else np.repeat(cfg["x"], 8, axis=0)
        self._io(x8, self.N)
        self.ws = T.workspace(T.tf_qlinear_workspace_bytes(w0, 8))
        self.sample_x = x8
        self.desc = proj_desc(kind, self.K, self.N, self.step_ms)

    def call(self, i, M, flags, x, out):
        if self.signs is not None:
            self.T.tf_qlinear_run_rht(self.copies[i], x, self.signs, out=out, ws=self.ws, flags=flags)
        else:
            self.T.tf_qlinear_run(self.copies[i], x, gamma=self.gamma, eps=self.eps, out=out, ws=self.ws, flags=flags)

    def sample_matrix(self):
        return self.w, 256 if self.K <= 2048 else 32, "the weight matrix"


class Step(Workload):
    """The per-token weight stream of a 28-layer dense decoder (d_model 1024, d_ff 3072,
    16 q / 8 kv heads of 128, tied readout 151,936), one M=1 and one M=8 step per bench step."""

    name = "step"
    kernel_key = "step_b4_l28_d1024"
    kernel = "stage kernels (one CTA per 16-row block), 4 per layer, + the readout's warp-worker kernel, chained with programmatic dependent launch"
    launches_per_call = 4 * 28 + 1

    def __init__(self, T, torch, l2_bytes):
        super().__init__(T, torch)
        from skinny_gemm_bit_gb300 import synth
        cfg = synth.decoder(M=8)
        self.cfg = cfg
        d = cfg["dims"]
        layers = []
        for L in cfg["layers"]:
            layers.append({k: (_pack(T, v) if k in ("qkv", "o", "gate", "up", "down") else _dev_bf16(torch, v))
                           for k, v in L.items()})
        self.dec = T.Decoder(layers, _dev_bf16(torch, cfg["final_norm"]), _pack(T, cfg["readout"]), d["d_model"],
                             d["d_ff"], d["q_dim"], d["kv_dim"], cfg["eps"])
        self.K, self.N, self.bits = d["d_model"], d["vocab"], 4
        self.per_call = self.dec.weight_bytes()
        self.copies = [self.dec]  # 335 MB per step: more than twice L2 already
        self.n_copies = 1
        self._io(cfg["x"], d["vocab"])
        self.ws = T.workspace(T.tf_decode_step_workspace_bytes(self.dec, 8))
        self.sample_x = cfg["x"]
        self.desc = STEP_DESC

    def call(self, i, M, flags, x, out):
        self.T.tf_decode_step_run(self.dec, x, out=out, ws=self.ws, flags=flags)

    def sample_matrix(self):
        return self.cfg["layers"][0]["qkv"], 256, "layer 0's QKV matrix"


class MoE(Workload):
    """MoE expert projection: M=8 rows, 128 experts, top-8, hidden 2048, intermediate 768."""

    step_ms = (8,)
    launches_per_call = 4

    def __init__(self, T, torch, l2_bytes, bits: int, code: str = "mlx"):
        super().__init__(T, torch)
        from skinny_gemm_bit_gb300 import synth
        nvfp4 = code == "nvfp4"
        cfg = synth.moe_layer(bits=bits, code=code)
        self.cfg = cfg
        self.name = "moe_nvfp4" if nvfp4 else f"moe{bits}"
        self.kernel_key = "moe_nvfp4" if nvfp4 else f"moe_b{bits}"
        what = "NVFP4" if nvfp4 else f"{bits}-bit"
        self.kernel = f"MoE layer ({what}): route, gate/up, down, combine"
        g, u, dn = _pack(T, cfg["gate"]), _pack(T, cfg["up"]), _pack(T, cfg["down"])
        self.logits = torch.from_numpy(cfg["logits"]).cuda()
        self.K, self.N, self.bits = 2048, 768, bits
        stack = g.buf.numel() + u.buf.numel() + dn.buf.numel()
        n = max(2, int(np.ceil(2 * l2_bytes / stack)) + 1)
        self.copies = [(g, u, dn)] + [tuple(_clone_qweight(T, w) for w in (g, u, dn)) for _ in range(n - 1)]
        self.n_copies = n
        self._io(cfg["x"], 2048)
        self.ws = T.workspace(T.tf_qmoe_workspace_bytes(g, u, dn, 8, 8))
        self.idx = torch.empty((8, 8), dtype=torch.int32, device="cuda")
        self.wts = torch.empty((8, 8), dtype=torch.float32, device="cuda")
        _, idx, _ = T.tf_qmoe_run(g, u, dn, self.logits, self.x[8], 8, ws=self.ws)
        torch.cuda.synchronize()
        distinct = len(np.unique(idx.cpu().numpy()))
        self.per_call = distinct * (g.weight_bytes() + u.weight_bytes() + dn.weight_bytes()) // 128
        self.sample_x = cfg["x"]
        self.desc = moe_desc(nvfp4, bits, distinct)

    def call(self, i, M, flags, x, out):
        g, u, dn = self.copies[i]
        self.T.tf_qmoe_run(g, u, dn, self.logits, x, 8, out=out, idx=self.idx, wts=self.wts, ws=self.ws,
                           flags=flags)

    def sample_matrix(self):
        import oracle
        return oracle.expert(self.cfg["gate"], 0), 128, "expert 0's gate matrix"


WORKLOADS = ("step", "gateup", "proj", "wide", "wide_rht", "readout", "moe4", "moe8", "moe_nvfp4", "verify",
             "wide_nvfp4", "readout_nvfp4")
PROJ_KINDS = ("proj", "wide", "wide_rht", "readout", "wide_nvfp4", "readout_nvfp4")


def make_workload(name, T, torch, l2_bytes):
    if name == "gateup":
        return GateUp(T, torch, l2_bytes)
    if name in PROJ_KINDS:
        return Proj(T, torch, l2_bytes, kind=name)
    if name == "step":
        return Step(T, torch, l2_bytes)
    if name in ("moe4", "moe8"):
        return MoE(T, torch, l2_bytes, bits=int(name[3]))
    if name == "moe_nvfp4":
        return MoE(T, torch, l2_bytes, bits=4, code="nvfp4")
    raise ValueError(name)


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
    wl = make_workload(args.workload, T, torch, l2)
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
    # five timed replays, each after an L2 flush (a buffer of twice L2 written, outside
    # the timed region): no call of a replay finds its weights in L2
    flush = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")
    replay_ms = []
    for _ in range(REPLAYS):
        flush.fill_(1)
        torch.cuda.synchronize()
        barrier(pg)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record()
        g_timed.replay()
        ev1.record()
        torch.cuda.synchronize()
        barrier(pg)
        replay_ms.append(max_over_ranks(ev0.elapsed_time(ev1), pg, f"cuda:{local}"))
    clocks = sampler.stop()
    ms_max = statistics.median(replay_ms)

    # end to end: host buffers in, host buffers out, inside the timed region
    g_e2e.replay()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(REPLAYS):
        flush.fill_(1)
        torch.cuda.synchronize()
        barrier(pg)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g_e2e.replay()
        e1.record()
        torch.cuda.synchronize()
        barrier(pg)
        e2e_ms.append(max_over_ranks(e0.elapsed_time(e1), pg, f"cuda:{local}"))
    ms_e2e = statistics.median(e2e_ms)

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
    call_us = ms_max * 1e3 / (K * len(wl.step_ms))
    achieved = wl.per_call / (call_us * 1e-6) / 1e9
    cpu = cpu_baseline(wl, args.cpu_seconds)
    h2d, d2h = wl.io_bytes()
    ms_list = sorted(set(wl.step_ms))
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms_max / K, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": f"synthetic (seeded random {_weights_word(wl)} weights and N(0,1) activations)",
        "config": {"workload": wl.desc, "name": wl.name, "K": wl.K, "N": wl.N, "M": ms_list, "bits": wl.bits,
                   "group": 64,
                   "l2": (f"L2 flushed (a buffer of twice L2 written) before each timed replay; the calls of a "
                          f"replay rotate over {wl.n_copies} weight copies ({wl.n_copies * wl.per_call / l2:.1f}x L2), "
                          f"so every call streams its weights from HBM"
                          if wl.n_copies > 1 else
                          f"L2 flushed before each timed replay; one copy of the weights, "
                          f"{wl.per_call / 1e6:.1f} MB per call ({wl.per_call / l2:.1f}x L2), streamed from HBM by "
                          f"every call"),
                   "timing": f"median of {REPLAYS} timed replays of the {K}-step graph: "
                             + ", ".join(f"{v:.4f}" for v in replay_ms) + " ms",
                   "graph": "CUDA graph" + (", programmatic dependent launch" if flags else ""),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_hbm_measured": round(100 * value / world / peak, 2),
        "pct_of_8tbs_nominal": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "per_m": {str(M): {"us_per_call": round(us, 3), "gbs": round(wl.per_call / (us * 1e-6) / 1e9, 1)}
                  for M, us in per_m.items()},
        "per_m_no_pdl": {str(M): {"us_per_call": round(us, 3), "gbs": round(wl.per_call / (us * 1e-6) / 1e9, 1)}
                         for M, us in per_m_nopdl.items()},
        "m8_over_m1": round(per_m[8] / per_m[1], 3) if 1 in per_m and 8 in per_m else None,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": recorded_traffic(wl.kernel_key),
                     "peak_source": peak_kind, "kernel": wl.kernel,
                     "bytes_per_launch": wl.per_call, "launch_us": round(call_us, 3)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": K * wl.launches_per_step,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def run_verify(args):
    """Greedy generation with the M = 8 verify block on the 28-layer decoder: a host-driven
    loop (one synchronisation a step), timed end to end with CUDA events around whole
    generations, against plain one-token decoding on the same prompt."""
    import torch
    world, rank, local, pg = dist_setup()
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    from skinny_gemm_bit_gb300 import tfq as T
    wl = Step(T, torch, 0)  # the full-size decoder; its descriptor and weights
    dec = wl.dec
    n_new = 64
    start = int(np.random.default_rng(5).integers(0, dec.readout.N))
    ws = T.workspace(T.tf_generate_workspace_bytes(dec))
    cont, _, _ = T.tf_generate_greedy(dec, [start], n_new, max_draft=0, ws=ws)
    prompt = [start] + cont[: 3 * n_new // 4] + [start]  # holds most of the continuation
    K, W = args.steps, args.warmup
    K = max(1, min(K, 20))  # a generation is ~20-40 ms: 20 of them time well within the budget

    def timed(max_draft):
        for _ in range(W):
            T.tf_generate_greedy(dec, prompt, n_new, max_draft=max_draft, ws=ws)
        torch.cuda.synchronize()
        barrier(pg)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        steps = acc = 0
        for _ in range(K):
            toks, st, ac = T.tf_generate_greedy(dec, prompt, n_new, max_draft=max_draft, ws=ws)
            steps, acc = steps + st, acc + ac
        e1.record()
        torch.cuda.synchronize()
        barrier(pg)
        return max_over_ranks(e0.elapsed_time(e1), pg, f"cuda:{local}"), steps, acc, toks

    sampler = ClockSampler(local)
    sampler.start()
    ms, steps, acc, toks = timed(7)
    clocks = sampler.stop()
    ms_plain, steps_plain, _, toks_plain = timed(0)
    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return
    assert toks == toks_plain, "the verify block changed the generated tokens"
    peak, peak_kind = measured_peaks()
    step_bytes = dec.weight_bytes()
    value = world * step_bytes * steps / (ms * 1e-3) / 1e9
    us_step = ms * 1e3 / steps
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms / K, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded random 4-bit weights; prompt from the model's own greedy output)",
        "config": {"workload": (f"greedy generation of {n_new} tokens with prompt-lookup drafts and an up-to-8-row "
                                f"verify block, 28-layer dense decoder d_model 1024, tied readout 151936; a bench step "
                                f"is one generation"),
                   "name": "verify", "tokens_per_generation": n_new, "prompt_len": len(prompt),
                   "decoder_steps_per_generation": round(steps / K, 2),
                   "drafts_kept_per_generation": round(acc / K, 2),
                   "tokens_per_s": round(world * n_new * K / (ms * 1e-3), 1),
                   "plain_tokens_per_s": round(world * n_new * K / (ms_plain * 1e-3), 1),
                   "plain_decoder_steps_per_generation": round(steps_plain / K, 2),
                   "us_per_decoder_step": round(us_step, 2),
                   "graph": "none (host-driven loop; one synchronisation per decoder step)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_hbm_measured": round(100 * value / world / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(step_bytes / (us_step * 1e-6) / 1e9, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(step_bytes / (us_step * 1e-6) / 1e9 / peak, 4),
                     "traffic": recorded_traffic("step_b4_l28_d1024"), "peak_source": peak_kind,
                     "kernel": "decoder step at M = 1 + drafts, embedding and argmax kernels",
                     "bytes_per_launch": step_bytes, "launch_us": round(us_step, 3)},
        "cpu_baseline": cpu_baseline(wl, args.cpu_seconds),
        "e2e": {"value": round(value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(4 * (steps + acc) / K), "d2h_bytes_per_step": int(36 * steps / K),
                "note": "the loop is host-driven: value is already end to end"},
        "gpu_launches": steps * (Step.launches_per_call + 2),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def cpu_model() -> str:
    """The host CPU's model name (from /proc/cpuinfo; lscpu's when that has none)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def cpu_baseline(wl, seconds):
    """The fp64 oracle on a bounded sample of the workload: on every host core at once
    (threads, each on its own slice of the sample's rows; the oracle's C loops release
    the interpreter lock) and on one thread."""
    cores = os.cpu_count() or 1
    done1, el1, desc1 = wl.oracle_sample(seconds / 2)
    results = [None] * cores
    def work(i):
        results[i] = wl.oracle_sample(seconds / 2, part=(i, cores))
    threads = [threading.Thread(target=work, args=(i,)) for i in range(cores)]
    t0 = time.perf_counter()
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    el = time.perf_counter() - t0
    done = sum(r[0] for r in results)
    return {"value": round(done / el / 1e9, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"{cores} threads, each on 1/{cores} of the rows of: {results[0][2]}",
            "single_thread": {"value": round(done1 / el1 / 1e9, 6), "unit": "GB/s", "sample": desc1}}


class _HostOnly:
    """The CPU side of a workload (its oracle sample), without packing anything on a GPU."""

    def __init__(self, name):
        from skinny_gemm_bit_gb300 import synth
        self.name = name
        if name == "gateup":
            self.impl = GateUp.__new__(GateUp)
            cfg = synth.fused_gateup(seed=1, M=8)
            self.impl.cfg, self.impl.K, self.impl.N = cfg, 1024, 3072
            self.desc = gateup_desc(1024, 3072)
            self.K, self.N, self.ms, self.bits = 1024, 3072, [1, 8], 4
        else:
            self.impl = Workload.__new__(Workload)
            if name in PROJ_KINDS:
                cfg = _proj_config(name)
                w = cfg["w"]
                x8 = cfg["x"] if cfg["x"].shape[0] == 8 else np.repeat(cfg["x"], 8, axis=0)
                rows, what = (256, "the weight matrix") if w["K"] <= 2048 else (32, "the weight matrix")
                self.impl.step_ms = (1,) if name == "proj" else (1, 8)
                if name == "wide_rht":
                    self.impl.host_signs = synth.rht_signs(np.random.default_rng(2), 12800)
                self.K, self.N, self.bits = w["K"], w["N"], 4
                self.desc = proj_desc(name, w["K"], w["N"], self.impl.step_ms)
            elif name in ("step", "verify"):
                cfg = synth.decoder(M=8, n_layers=1)  # layer 0 of the same seeded model
                w, x8, rows, what = cfg["layers"][0]["qkv"], cfg["x"], 256, "layer 0's QKV matrix"
                self.impl.step_ms = (1, 8)
                self.K, self.N, self.bits = 1024, 151936, 4
                self.desc = STEP_DESC
            else:
                import oracle
                nvfp4 = name == "moe_nvfp4"
                bits = 4 if nvfp4 else int(name[3])
                cfg = synth.moe_layer(code="nvfp4") if nvfp4 else synth.moe_layer(bits=bits)
                w = oracle.expert(cfg["gate"], 0)
                x8, rows, what = cfg["x"], 128, "expert 0's gate matrix"
                self.impl.step_ms = (8,)
                self.K, self.N, self.bits = 2048, 768, bits
                idx, _ = oracle.topk_softmax(cfg["logits"], cfg["top_k"])
                self.desc = moe_desc(nvfp4, bits, len(np.unique(idx)))
            self.impl.sample_x = x8
            self.impl.sample_matrix = lambda w=w, rows=rows, what=what: (w, rows, what)
            self.ms = sorted(set(self.impl.step_ms))

    def oracle_sample(self, seconds, part=(0, 1)):
        if self.name == "gateup":
            return GateUp.oracle_sample(self.impl, seconds, part)
        return Workload.oracle_sample(self.impl, seconds, part)


def run_reference(args):
    """The fp64 oracle as the reference arm, on this host's cores, rank 0 only."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    host = _HostOnly(args.workload)
    cores = os.cpu_count() or 1
    desc = None
    steps_s = []
    for i in range(args.warmup + args.steps):
        results = [None] * cores

        def work(j):
            results[j] = host.oracle_sample(args.ref_step_seconds, part=(j, cores))
        threads = [threading.Thread(target=work, args=(j,)) for j in range(cores)]
        t0 = time.perf_counter()
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        el = time.perf_counter() - t0
        desc = f"{cores} threads, each on 1/{cores} of the rows of: {results[0][2]}"
        if i >= args.warmup:
            steps_s.append((sum(r[0] for r in results), el))
    total_b = sum(d for d, _ in steps_s)
    total_s = sum(e for _, e in steps_s)
    value = total_b / total_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total_s / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": f"synthetic (seeded random {_weights_word(host)} weights and N(0,1) activations)",
        "config": {"workload": host.desc, "name": host.name, "K": host.K, "N": host.N, "M": host.ms,
                   "bits": host.bits, "group": 64},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "kind": "oracle", "cores": cores,
                         "cpu": cpu_model(), "sample": f"each step: {desc}"},
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
    ap.add_argument("--workload", default="step", choices=WORKLOADS,
                    help="step (default): 28-layer decoder weight stream, M=1 and 8; gateup: fused RMSNorm + "
                         "gate/up, K=1024, N=2x3072, M=1 and 8; proj: "
                         "K=1024, N=3072, M=1; wide: K=12800, N=2560, M=1 and 8; wide_rht: the same with the "
                         "input Hadamard transform; readout: RMSNorm + tied "
                         "readout, K=1024, N=151936, M=1 and 8; "
                         "moe4 / moe8 / moe_nvfp4: MoE layer, M=8 (4-bit, 8-bit, NVFP4 experts); verify: greedy generation with prompt-lookup drafts and "
                         "an up-to-8-row verify block on the 28-layer decoder; wide_nvfp4 / readout_nvfp4: the "
                         "wide and readout shapes with NVFP4 weights")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "verify":
        run_verify(args)
    else:
        run_tfq(args)


if __name__ == "__main__":
    main()
