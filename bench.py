"""Benchmark of the mLSTM cell forward on one B300 (or N, one process per GPU).

A step is one chunkwise forward of the 1.3B-style layer (B=4, NH=4, S=2048, d=512, chunk 64,
bf16 q/k/v, fp32 gates, fp32 h) through the library's mlstm_fwd_chunkwise: on the tensor-core
path that is a single fused kernel (gate preprocessing, state passing and output).  The decode
step (B=256, NH=8, d=256, fp32 state) is timed in its own loop and reported under "decode".
Inputs are synthetic (seeded) and resident in HBM; L2 is flushed between timed iterations (a
256 MiB write) outside the timed events.  SM clocks and throttle reasons are sampled during the
timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle on a bounded
sample of the same workload instead (the reference arm of this build).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mlstm_matrix_memory_02_b300 import workloads as W  # noqa: E402

FWD = W.LAYER_1P3B
DEC = W.DECODE


def fwd_flops(w) -> float:
    """Algorithmic flops of one chunkwise forward: per head and chunk, L(L+1)(dqk+dv) for the
    causal Q K^T and (S o D) V, plus 4 L dqk dv for Q C^T and the state update."""
    L = w.chunk
    per_chunk = L * (L + 1) * (w.DQK + w.DV) + 4 * L * w.DQK * w.DV
    return float(per_chunk * (w.S // L) * w.B * w.NH)


def fwd_bytes(w, h_bytes=4) -> float:
    """Algorithmic HBM bytes: q, k, v read once (bf16), gates read once, h written once,
    final state written once."""
    P = w.B * w.NH
    qkv = P * w.S * (2 * w.DQK + w.DV) * 2
    gates = P * w.S * 2 * 4
    h = P * w.S * w.DV * h_bytes
    state = P * (w.DV * w.DQK + w.DQK + 1) * 4
    return float(qkv + gates + h + state)


def dec_bytes(w, h_bytes=4) -> float:
    """Algorithmic bytes of one decode step: C and n read and written, m read and written,
    q, k, v (bf16) and the gates read, h written."""
    P = w.B * w.NH
    return float(P * (2 * w.DV * w.DQK * 4 + 2 * w.DQK * 4 + 2 * 4
                      + (2 * w.DQK + w.DV) * 2 + 2 * 4 + w.DV * h_bytes))


def captured_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` (an entry of profiles/traffic.json: a kernel name, or
    forward@workload / backward@workload for a call of several kernels) from the committed ncu
    summary, or None when one of its sources has changed since that capture (the entry holds a
    hash of the listed source files)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entry = json.load(f).get(kernel)
    if not entry:
        return None
    h = hashlib.sha256()
    for src in entry.get("sources", [entry.get("source")]):
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return float(entry["dram_bytes"]) if h.hexdigest()[:16] == entry["sha"] else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


_NVML_LOOP = r"""
import ctypes, sys, time
nvml = ctypes.CDLL("libnvidia-ml.so.1")
assert nvml.nvmlInit_v2() == 0
h = ctypes.c_void_p()
assert nvml.nvmlDeviceGetHandleByIndex_v2(int(sys.argv[1]), ctypes.byref(h)) == 0
period = float(sys.argv[2])
try:
    reasons_fn = nvml.nvmlDeviceGetCurrentClocksEventReasons
except AttributeError:
    reasons_fn = nvml.nvmlDeviceGetCurrentClocksThrottleReasons
sm, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
print("ready", flush=True)
while True:
    nvml.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm))      # NVML_CLOCK_SM
    nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
    reasons_fn(h, ctypes.byref(rs))
    print(time.time(), sm.value, mx.value, rs.value, flush=True)
    time.sleep(period)
"""


class ClockSampler:
    """SM clocks and throttle reasons sampled about every millisecond while the timed region
    runs, by a separate process calling the NVML library directly (nvidia-smi at 200 ms if that
    fails); only the samples taken inside the timed region are summarised."""

    REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "sw_power_cap": 0x4}

    def __init__(self, gpu_index: int, period_s: float = 0.001):
        self.gpu = gpu_index
        self.period = period_s
        self.samples = []  # (sm_mhz, max_mhz, reasons bitmask, wall time)
        self.window = None
        self.proc = None
        self.kind = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen([sys.executable, "-c", _NVML_LOOP, str(self.gpu), str(self.period)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            first = self.proc.stdout.readline()
            if first.strip() != "ready":
                raise RuntimeError("nvml sampler did not start")
            self.kind = "nvml"
        except Exception:  # noqa: BLE001
            if self.proc is not None:
                self.proc.kill()
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.gpu}",
                     "--query-gpu=timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                     "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                     "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "200"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.kind = "nvidia-smi"
            except OSError:
                self.proc = None
        return self

    def mark(self, t0, t1):
        self.window = (t0, t1)  # wall-clock time.time() bounds of the timed region

    def __exit__(self, *exc):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for ln in out.splitlines():
            try:
                if self.kind == "nvml":
                    t, sm, mx, rs = ln.split()
                    self.samples.append((float(sm), float(mx), int(rs), float(t)))
                else:
                    parts = [x.strip() for x in ln.split(",")]
                    bits = [0x8, 0x40, 0x20, 0x4]
                    mask = sum(b for b, v in zip(bits, parts[3:7]) if v.lower() == "active")
                    self.samples.append((float(parts[1]), float(parts[2]), mask, None))
            except (ValueError, IndexError):
                continue

    def summary(self):
        sel, where = self.samples, "timed region"
        if self.window is not None and self.kind == "nvml":
            inside = [x for x in self.samples if self.window[0] <= x[3] <= self.window[1]]
            if inside:
                sel = inside
            else:
                where = "around the timed region (none fell inside it)"
        elif self.kind != "nvml":
            where = "while the timed region ran (nvidia-smi, 200 ms)"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        reasons = sorted(name for name, bit in self.REASONS.items() if any(x[2] & bit for x in sel))
        return {"sm_mhz": statistics.median(x[0] for x in sel), "sm_max_mhz": max(x[1] for x in sel),
                "reasons": reasons, "samples": len(sel), "sampled": where}


def dist_setup(timeout_s: float | None = None):
    """Process group from the torchrun environment.  Collectives (the barriers and the timing
    reduction) give up after `timeout_s` (default 600 s, or MLSTM_PG_TIMEOUT_S), so that a rank
    that died or never joined ends the others with an error instead of holding their GPUs."""
    import datetime

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if timeout_s is None:
            timeout_s = float(os.environ.get("MLSTM_PG_TIMEOUT_S", "600"))
        dist.init_process_group(backend=backend, timeout=datetime.timedelta(seconds=timeout_s))
    return rank, local, world


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------------ CPU oracle arm
def oracle_sample(w, heads: int):
    """The first `heads` (batch, head) pairs of the workload, for the CPU oracle."""
    inp = W.make_inputs(w.with_(B=1, NH=heads) if heads <= w.NH else w)
    if heads > w.NH:
        inp = {k: v.reshape(1, -1, *v.shape[2:])[:, :heads] for k, v in inp.items()}
    return inp


def time_oracle(w, heads: int, reps: int = 1, s_len: int = None):
    """Wall time of the oracle over `heads` head-sequences of workload w (the first s_len tokens
    of each, default all); tokens/s of the full layer (each layer token needs NH head-tokens)."""
    import oracle
    s_len = s_len or w.S
    inp = oracle_sample(w, heads)
    inp = {key: val[:, :, :s_len] for key, val in inp.items()}
    oracle.load()
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.recurrent(**inp)
        times.append(time.perf_counter() - t0)
    cores = min(os.cpu_count() or 1, heads)
    tps = heads * s_len / w.NH / statistics.median(times)
    return tps, cores, times


def run_reference(args, rank, world):
    if rank != 0:
        return
    heads = max(1, min(os.cpu_count() or 1, FWD.B * FWD.NH))
    # each step is a bounded sample: every thread gets one head, and the sequence prefix is sized
    # so that warm-up plus timed steps stay within about two and a half minutes
    budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    _, _, t_cal = time_oracle(FWD, heads, s_len=min(FWD.S, 4 * FWD.chunk))
    per_token = t_cal[0] / min(FWD.S, 4 * FWD.chunk)
    s_len = int(min(FWD.S, max(FWD.chunk, budget / max(per_token, 1e-9))) // FWD.chunk * FWD.chunk)
    for _ in range(args.warmup):
        time_oracle(FWD, heads, s_len=s_len)
    tps, cores, times = time_oracle(FWD, heads, reps=args.steps, s_len=s_len)
    value = tps
    sample = (f"{heads} of {FWD.B * FWD.NH} (batch, head) sequences of the {FWD.name}, first {s_len} of "
              f"S={FWD.S} tokens each, per step; tokens/s scaled to the whole layer (x 1/NH)")
    line = {
        "metric": "mLSTM chunkwise forward tokens/s (1.3B-style layer)", "value": value,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": FWD.name, "B": FWD.B, "NH": FWD.NH, "S": FWD.S, "DQK": FWD.DQK,
                   "DV": FWD.DV, "chunk": FWD.chunk, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ GPU arm
def time_layer(B, w, dev, args, flush, peaks):
    """One more forward workload, timed like the headline (L2 flushed between calls, CUDA events
    around each call), with h in the dtype of v (bf16) as the layer hands it on.  The 350M-style
    layer is HBM-bound (its roofline is HBM of algorithmic bytes); the long-context layer runs in
    sequence segments on the tensor-core path (6 launches: segment init, gate preprocessing,
    weights and tensor-core state walk of the first pass, scan, fused kernel) and is reported
    against HBM as well, with its tensor-core fraction beside it."""
    import torch
    inp = W.make_inputs(w)
    q, k, v = (torch.from_numpy(inp[x]).to(dev).to(torch.bfloat16) for x in ("q", "k", "v"))
    ig, fg = (torch.from_numpy(inp[x]).to(dev) for x in ("ig", "fg"))
    del inp
    out = (torch.empty((w.B, w.NH, w.S, w.DV), dtype=torch.bfloat16, device=dev),
           torch.empty((w.B, w.NH, w.DV, w.DQK), dtype=torch.float32, device=dev),
           torch.empty((w.B, w.NH, w.DQK), dtype=torch.float32, device=dev),
           torch.empty((w.B, w.NH), dtype=torch.float32, device=dev))
    ws = B.alloc_workspace(w.B, w.NH, w.S, w.DQK, w.DV, w.chunk, torch.bfloat16, dev)
    stream = torch.cuda.current_stream()

    def call():
        B.mlstm_fwd_chunkwise(q, k, v, ig, fg, w.chunk, h_dtype=torch.bfloat16, out=out, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    reps = max(args.steps, 5)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    l0 = B.mlstm_kernel_launches()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    launches = B.mlstm_kernel_launches() - l0
    B.mlstm_fwd_check(ws, w.B, w.NH, w.S, w.DQK, w.DV, w.chunk)
    us = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
    nbytes, flops = fwd_bytes(w, h_bytes=2), fwd_flops(w)
    gbs = nbytes / (us * 1e-6) / 1e9
    tf = flops / (us * 1e-6) / 1e12
    G = B.mlstm_fwd_segments(w.B, w.NH, w.S, w.DQK, w.DV, w.chunk)
    key = {W.LAYER_350M.name: "350m", W.STRESS_16K.name: "stress"}[w.name]
    return {"metric": f"mLSTM chunkwise forward tokens/s ({w.name})", "value": w.B * w.S / (us * 1e-6),
            "unit": "tokens/s", "us_per_launch": us,
            "config": {"workload": w.name, "B": w.B, "NH": w.NH, "S": w.S, "DQK": w.DQK, "DV": w.DV,
                       "chunk": w.chunk, "qkv": "bf16", "gates": "fp32", "h": "bf16",
                       "sequence_segments": G,
                       "l2": "flushed between timed calls (256 MiB write, outside the events)"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"],
                         "traffic": captured_traffic(f"forward@{key}"),
                         "kernel": ("fwd_tc_kernel (one launch)" if G == 1 else
                                    f"whole forward in {G} segments: seg_init, gates, state_weights, "
                                    "states_tc (first pass), seg_scan, fwd_tc_kernel"),
                         "algorithmic_bytes_per_launch": nbytes,
                         "peak_source": peaks["source"] + " HBM copy",
                         "tensor_tflops": tf, "tensor_frac": tf / peaks["bf16_tflops"]},
            "gpu_launches": int(launches)}


def time_backward(B, w, dev, args, flush, peaks):
    """The chunkwise backward (mlstm_bwd_chunkwise) of a layer for a random upstream gradient,
    bf16 q/k/v/dh and gradients, L2 flushed between calls.  Reported against the tensor-core
    peak with twice the forward's algorithmic flops (the usual backward-to-forward ratio of a
    layer built from products: each forward product has two gradient products)."""
    import torch
    inp = W.make_inputs(w)
    q, k, v = (torch.from_numpy(inp[x]).to(dev).to(torch.bfloat16) for x in ("q", "k", "v"))
    ig, fg = (torch.from_numpy(inp[x]).to(dev) for x in ("ig", "fg"))
    del inp
    g = torch.Generator(device=dev).manual_seed(21)
    dh = torch.randn((w.B, w.NH, w.S, w.DV), device=dev, generator=g).to(torch.bfloat16)
    ws = torch.empty(B.mlstm_bwd_workspace_bytes(w.B, w.NH, w.S, w.DQK, w.DV, w.chunk), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        B.mlstm_bwd_chunkwise(q, k, v, ig, fg, dh, w.chunk, workspace=ws)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(5)]
    l0 = B.mlstm_kernel_launches()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        B.mlstm_bwd_chunkwise(q, k, v, ig, fg, dh, w.chunk, workspace=ws)
        b.record(stream)
    torch.cuda.synchronize()
    launches = B.mlstm_kernel_launches() - l0
    B.mlstm_fwd_check(ws, w.B, w.NH, w.S, w.DQK, w.DV, w.chunk)  # the error word sits at offset 0 here too
    us = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
    flops = 2 * fwd_flops(w)
    tf = flops / (us * 1e-6) / 1e12
    return {"metric": f"mLSTM chunkwise backward tokens/s ({w.name})", "value": w.B * w.S / (us * 1e-6),
            "unit": "tokens/s", "us_per_launch": us,
            "config": {"workload": w.name, "B": w.B, "NH": w.NH, "S": w.S, "DQK": w.DQK, "DV": w.DV,
                       "chunk": w.chunk, "qkv_dh_grads": "bf16", "gates": "fp32",
                       "state_walks": "tensor cores (tcgen05)", "chunk_products": "CUDA cores, fp32",
                       "l2": "flushed between timed calls"},
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16_tflops"], "traffic": captured_traffic("backward@350m"),
                         "algorithmic_flops_per_launch": flops,
                         "kernel": "whole backward (gates, state walks, output recompute, chunk gradients)",
                         "peak_source": f"{peaks['source']} bf16 dense (burst)"},
            "gpu_launches": int(launches)}


def run_ours(args, rank, local, world):
    import torch
    from mlstm_matrix_memory_02_b300 import binding as B

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    w = FWD

    inp = W.make_inputs(w)
    q = torch.from_numpy(inp["q"]).to(dev).to(torch.bfloat16)
    k = torch.from_numpy(inp["k"]).to(dev).to(torch.bfloat16)
    v = torch.from_numpy(inp["v"]).to(dev).to(torch.bfloat16)
    ig = torch.from_numpy(inp["ig"]).to(dev)
    fg = torch.from_numpy(inp["fg"]).to(dev)
    P = w.B * w.NH
    h = torch.empty((w.B, w.NH, w.S, w.DV), dtype=torch.float32, device=dev)
    C = torch.empty((w.B, w.NH, w.DV, w.DQK), dtype=torch.float32, device=dev)
    n = torch.empty((w.B, w.NH, w.DQK), dtype=torch.float32, device=dev)
    m = torch.empty((w.B, w.NH), dtype=torch.float32, device=dev)
    ws = B.alloc_workspace(w.B, w.NH, w.S, w.DQK, w.DV, w.chunk, torch.bfloat16, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        B.mlstm_fwd_chunkwise(q, k, v, ig, fg, w.chunk, h_dtype=torch.float32, out=(h, C, n, m), workspace=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    launches0 = B.mlstm_kernel_launches()
    with ClockSampler(local) as clk:
        t_start = time.time()
        for i in range(args.steps):
            flush.zero_()  # evict the inputs from L2 (outside the timed events)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        clk.mark(t_start, time.time())
    launches_fwd = B.mlstm_kernel_launches() - launches0
    barrier(world)
    step_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, world)
    tokens = w.B * w.S
    value = tokens * world / (ms_max * 1e-3)

    flops = fwd_flops(w)
    path = B.mlstm_fwd_path(w.B, w.NH, w.S, w.DQK, w.DV, w.chunk)
    per_step = launches_fwd / max(args.steps, 1)
    five = path >= 1 and round(per_step) == 5  # gate chain, pre-pass, n chain, denominators, state walk
    achieved_tf = flops / (ms * 1e-3) / 1e12
    # the same forward through the single fused kernel (the least workspace selects it), for context
    ws_least = torch.empty(B.mlstm_fwd_workspace_min_bytes(w.B, w.NH, w.S, w.DQK, w.DV, w.chunk),
                           dtype=torch.uint8, device=dev)
    fused_ms = None
    if five:
        for _ in range(3):
            B.mlstm_fwd_chunkwise(q, k, v, ig, fg, w.chunk, h_dtype=torch.float32, out=(h, C, n, m),
                                  workspace=ws_least)
        fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
        for a_, b_ in fev:
            flush.zero_()
            a_.record(stream)
            B.mlstm_fwd_chunkwise(q, k, v, ig, fg, w.chunk, h_dtype=torch.float32, out=(h, C, n, m),
                                  workspace=ws_least)
            b_.record(stream)
        torch.cuda.synchronize()
        fused_ms = statistics.median(a_.elapsed_time(b_) for a_, b_ in fev)
    roofline = {"bound": "tensor", "achieved": achieved_tf, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved_tf / peaks["bf16_tflops"],
                # the committed capture is of the 1.3B-style layer: other workloads report none
                "traffic": (captured_traffic("forward@1p3b" if five else "fwd_tc_kernel")
                            if path >= 1 and w is W.LAYER_1P3B else None),
                "kernel": ("the whole forward call, five launches: gate chain, pre-pass (Q K^T on tensor "
                           "cores, P, beta q, w k), n chain, denominators, state walk (U, X, P V on tensor "
                           "cores; the largest share)" if five else
                           "fwd_tc_kernel (the whole forward: one launch)" if path >= 1
                           else "gates + states + output kernels"),
                "fused_single_kernel_ms": fused_ms,
                "algorithmic_flops_per_launch": flops, "ms_per_launch": ms,
                "peak_source": f"{peaks['source']} bf16 dense (burst); fp16 operands run at the same rate",
                "frac_of_sustained": achieved_tf / peaks["bf16_tflops_sustained"]
                if peaks.get("bf16_tflops_sustained") else None,
                "hbm_gbs_of_algorithmic_bytes": fwd_bytes(w) / (ms * 1e-3) / 1e9,
                "hbm_frac_of_algorithmic_bytes": fwd_bytes(w) / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}

    # ---- decode step: B=256, NH=8, d=256 state from a 512-token prefill through the library
    dw = DEC
    prior, steps = W.make_decode_inputs(dw.with_(S=max(args.steps, 16)))
    dq = torch.from_numpy(prior["q"]).to(dev).to(torch.bfloat16)
    dk = torch.from_numpy(prior["k"]).to(dev).to(torch.bfloat16)
    dv = torch.from_numpy(prior["v"]).to(dev).to(torch.bfloat16)
    _, Cd, nd, md = B.mlstm_fwd_chunkwise(dq, dk, dv, torch.from_numpy(prior["ig"]).to(dev),
                                          torch.from_numpy(prior["fg"]).to(dev), 64,
                                          h_dtype=torch.float32)
    del dq, dk, dv
    sq = torch.from_numpy(steps["q"]).to(dev).to(torch.bfloat16)
    sk = torch.from_numpy(steps["k"]).to(dev).to(torch.bfloat16)
    sv = torch.from_numpy(steps["v"]).to(dev).to(torch.bfloat16)
    sig = torch.from_numpy(steps["ig"]).to(dev)
    sfg = torch.from_numpy(steps["fg"]).to(dev)
    per_step = [tuple(x[:, :, t].contiguous() for x in (sq, sk, sv, sig, sfg)) for t in range(sq.shape[2])]
    hd = torch.empty((dw.B, dw.NH, dw.DV), dtype=torch.float32, device=dev)
    for t in range(max(args.warmup, 3)):
        B.mlstm_step(*per_step[t % len(per_step)], Cd, nd, md, h=hd)
    torch.cuda.synchronize()
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    launches1 = B.mlstm_kernel_launches()
    d0.record(stream)
    for t in range(args.steps):  # the 512 MiB state is far larger than L2
        B.mlstm_step(*per_step[t % len(per_step)], Cd, nd, md, h=hd)
    d1.record(stream)
    torch.cuda.synchronize()
    launches_dec = B.mlstm_kernel_launches() - launches1
    P_dec = dw.B * dw.NH
    dec_ms = d0.elapsed_time(d1) / max(args.steps, 1)
    dec_gbs = dec_bytes(dw) / (dec_ms * 1e-3) / 1e9
    # multi-token decode: T tokens per launch, the state crosses HBM once per launch
    multi = {}
    for T in (4, 8, 16):
        mq, mk, mv = (x[:, :, :T].contiguous() for x in (sq, sk, sv))
        mig, mfg = sig[:, :, :T].contiguous(), sfg[:, :, :T].contiguous()
        hm = torch.empty((dw.B, dw.NH, T, dw.DV), dtype=torch.float32, device=dev)
        for _ in range(max(args.warmup, 3)):
            B.mlstm_step_multi(mq, mk, mv, mig, mfg, Cd, nd, md, h=hm)
        torch.cuda.synchronize()
        reps = max(4, args.steps // T)
        m0 = torch.cuda.Event(enable_timing=True)
        m1 = torch.cuda.Event(enable_timing=True)
        l0 = B.mlstm_kernel_launches()
        m0.record(stream)
        for _ in range(reps):
            B.mlstm_step_multi(mq, mk, mv, mig, mfg, Cd, nd, md, h=hm)
        m1.record(stream)
        torch.cuda.synchronize()
        launches_dec += B.mlstm_kernel_launches() - l0
        us = m0.elapsed_time(m1) / reps * 1e3
        state_bytes = float(P_dec * 2 * dw.DV * dw.DQK * 4)
        tok_bytes = float(P_dec * T * ((2 * dw.DQK + dw.DV) * 2 + 2 * 4 + dw.DV * 4))
        multi[f"T{T}"] = {"us_per_launch": us, "tokens_per_s": dw.B * T / (us * 1e-6),
                          "speedup_vs_single_step": (dec_ms * 1e3 * T) / us,
                          "effective_gbs": (state_bytes + tok_bytes) / (us * 1e-6) / 1e9,
                          "frac_of_hbm": (state_bytes + tok_bytes) / (us * 1e-6) / 1e9 / peaks["hbm_gbs"]}
    decode = {"metric": "mLSTM decode step GB/s (B=256, NH=8, d=256, fp32 state)",
              "value": dec_gbs, "unit": "GB/s", "us_per_step": dec_ms * 1e3,
              "tokens_per_s": dw.B / (dec_ms * 1e-3),
              "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": dec_gbs / peaks["hbm_gbs"],
                           "traffic": captured_traffic("step_kernel"),
                           "kernel": "mlstm_step", "algorithmic_bytes_per_launch": dec_bytes(dw),
                           "peak_source": peaks["source"] + " HBM copy"},
              "frac_of_nominal_8tbs": dec_gbs / 8000.0,
              "multi_token": multi}
    del Cd, nd, md

    # ---- block step after the cell: group norm + output gate on the layer's h (fp32 h, bf16
    # o~ and y: 134 MB per launch, larger than L2, so consecutive launches do not hit in L2)
    g_rng = torch.Generator(device=dev).manual_seed(3)
    o_pre = torch.randn(h.shape, device=dev, generator=g_rng).to(torch.bfloat16)
    gam = 1.0 + 0.3 * torch.randn((w.NH, w.DV), device=dev, generator=g_rng)
    bet = 0.2 * torch.randn((w.NH, w.DV), device=dev, generator=g_rng)
    y_gn = torch.empty(h.shape, dtype=torch.bfloat16, device=dev)
    for _ in range(max(args.warmup, 3)):
        B.mlstm_groupnorm_gate(h, o_pre, gam, bet, 1e-5, out=y_gn)
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    l0 = B.mlstm_kernel_launches()
    g0.record(stream)
    for _ in range(args.steps):
        B.mlstm_groupnorm_gate(h, o_pre, gam, bet, 1e-5, out=y_gn)
    g1.record(stream)
    torch.cuda.synchronize()
    launches_gn = B.mlstm_kernel_launches() - l0
    gn_us = g0.elapsed_time(g1) / max(args.steps, 1) * 1e3
    gn_bytes = float(h.numel() * (4 + 2 + 2) + 2 * w.NH * w.DV * 4)
    gn_gbs = gn_bytes / (gn_us * 1e-6) / 1e9
    block_epilogue = {"metric": "group norm + output gate GB/s (1.3B-style layer h: fp32 in, bf16 o~ and y)",
                      "value": gn_gbs, "unit": "GB/s", "us_per_launch": gn_us,
                      "roofline": {"bound": "hbm", "achieved": gn_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                   "frac": gn_gbs / peaks["hbm_gbs"],
                                   "traffic": captured_traffic("groupnorm_gate_kernel"),
                                   "kernel": "groupnorm_gate_kernel", "algorithmic_bytes_per_launch": gn_bytes,
                                   "peak_source": peaks["source"] + " HBM copy"},
                      "l2": "134 MB per launch, larger than L2 (no flush)"}
    del o_pre, y_gn

    # ---- the other forward workloads: the 350M-style layer and the long-context layer
    layers = {"layer_350m": time_layer(B, W.LAYER_350M, dev, args, flush, peaks),
              "stress": time_layer(B, W.STRESS_16K, dev, args, flush, peaks),
              "backward_350m": time_backward(B, W.LAYER_350M, dev, args, flush, peaks)}

    # ---- end to end through the public API: pinned host inputs in, h back to the host, every
    # step.  Two streams take alternate steps, each with its own device inputs, outputs, workspace
    # and pinned host output, so a step's upload overlaps the previous step's download (PCIe
    # carries both directions at once); within a stream a step waits for the previous use of its
    # buffers.  Each step also flushes L2 (a 256 MiB write) inside the timed region.
    pin = {key: torch.from_numpy(inp[key]).to(torch.bfloat16 if key in "qkv" else torch.float32).pin_memory()
           for key in ("q", "k", "v", "ig", "fg")}
    nbuf = 2
    streams = [torch.cuda.Stream(device=dev) for _ in range(nbuf)]
    dbufs = [{key: torch.empty(t.shape, dtype=t.dtype, device=dev) for key, t in pin.items()} for _ in range(nbuf)]
    outs = [(torch.empty_like(h), torch.empty_like(C), torch.empty_like(n), torch.empty_like(m)) for _ in range(nbuf)]
    wss = [ws] + [B.alloc_workspace(w.B, w.NH, w.S, w.DQK, w.DV, w.chunk, torch.bfloat16, dev) for _ in range(nbuf - 1)]
    h_hosts = [torch.empty(h.shape, dtype=torch.float32).pin_memory() for _ in range(nbuf)]
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = h_hosts[0].numel() * h_hosts[0].element_size()

    def e2e_step(i):
        j = i % nbuf
        with torch.cuda.stream(streams[j]):
            flush.zero_()
            for key, t in pin.items():
                dbufs[j][key].copy_(t, non_blocking=True)
            d_ = dbufs[j]
            B.mlstm_fwd_chunkwise(d_["q"], d_["k"], d_["v"], d_["ig"], d_["fg"], w.chunk, h_dtype=torch.float32,
                                  out=outs[j], workspace=wss[j], stream=streams[j])
            h_hosts[j].copy_(outs[j][0], non_blocking=True)

    for i in range(max(args.warmup, 3)):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for st in streams:
        st.wait_stream(stream)
    for i in range(args.steps):
        e2e_step(i)
    for st in streams:
        stream.wait_stream(st)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = [e0.elapsed_time(e1) / args.steps]
    e2e_val = tokens * world / (max_over_ranks(statistics.mean(e2e_ms), world) * 1e-3)

    if rank != 0:
        return
    line = {
        "metric": f"mLSTM chunkwise forward tokens/s ({w.name})",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "NH": w.NH, "S": w.S, "DQK": w.DQK, "DV": w.DV,
                   "chunk": w.chunk, "qkv": "bf16", "gates": "fp32", "h": "fp32",
                   "mma": "fp16 operands (bf16 for Q K^T), fp32 accumulation in tensor memory",
                   "kernel_path": ("tensor cores (tcgen05): five kernels, the per-chunk work once per head and "
                                   "chunk (pre-pass), the state walk with d_qk split over a CTA pair" if five else
                                   {0: "CUDA cores", 1: "tensor cores (tcgen05, fused, one CTA per d_v tile)",
                                    2: "tensor cores (tcgen05, fused, d_qk split over a CTA pair)"}[path]),
                   "l2": "flushed between timed iterations (256 MiB write, outside the events)",
                   "per_rank": "each rank runs the full layer batch (weak scaling)"},
        "roofline": roofline,
        "decode": decode,
        "block_epilogue": block_epilogue,
        "layer_350m": layers["layer_350m"],
        "stress": layers["stress"],
        "backward_350m": layers["backward_350m"],
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "pipelining": "two streams take alternate steps (own inputs, outputs, workspace): a step's "
                              "upload overlaps the previous step's download; L2 flushed every step"},
        "gpu_launches": int(launches_fwd),
        "gpu_launches_other": {"decode": int(launches_dec), "block_epilogue": int(launches_gn),
                               "layer_350m": layers["layer_350m"]["gpu_launches"],
                               "stress": layers["stress"]["gpu_launches"],
                               "backward_350m": layers["backward_350m"]["gpu_launches"]},
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        heads = max(1, min(os.cpu_count() or 1, P))
        tps, cores, times = time_oracle(w, heads)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"{heads} of {P} (batch, head) sequences of the {w.name}, "
                                          f"full S={w.S}; tokens/s scaled to the layer (x 1/NH)",
                                "seconds": times[0]}
    print(json.dumps(line), flush=True)


def run_profile(kind: str):
    """Small, self-contained launches for ncu captures: one warm-up and one timed-shape call.

    fwd:          the --workload forward (one fused launch on the tensor-core path; four for the
                  long-context layer in sequence segments)
    decode:       one decode step of the B=256, NH=8, d=256 state (state initialised randomly)
    decode_multi: 16 decode steps in one launch on the same state
    gn:           group norm + output gate on a 1.3B-layer-shaped h (fp32 h, bf16 o~ and y)
    bwd:          the chunkwise backward of the 350M-style layer (bf16)"""
    import torch
    from mlstm_matrix_memory_02_b300 import binding as B
    dev = torch.device("cuda", 0)
    if kind == "fwd":
        w = FWD
        inp = W.make_inputs(w)
        q, k, v = (torch.from_numpy(inp[x]).to(dev).to(torch.bfloat16) for x in ("q", "k", "v"))
        ig, fg = (torch.from_numpy(inp[x]).to(dev) for x in ("ig", "fg"))
        # h as the bench writes it: fp32 for the 1.3B-style layer, bf16 for the others
        h_dtype = torch.float32 if w is W.LAYER_1P3B else torch.bfloat16
        for _ in range(2):
            B.mlstm_fwd_chunkwise(q, k, v, ig, fg, w.chunk, h_dtype=h_dtype)
    elif kind == "bwd":
        w = W.LAYER_350M
        inp = W.make_inputs(w)
        q, k, v = (torch.from_numpy(inp[x]).to(dev).to(torch.bfloat16) for x in ("q", "k", "v"))
        ig, fg = (torch.from_numpy(inp[x]).to(dev) for x in ("ig", "fg"))
        g = torch.Generator(device=dev).manual_seed(21)
        dh = torch.randn((w.B, w.NH, w.S, w.DV), device=dev, generator=g).to(torch.bfloat16)
        for _ in range(2):
            B.mlstm_bwd_chunkwise(q, k, v, ig, fg, dh, w.chunk)
    elif kind == "gn":
        w = FWD
        g = torch.Generator(device=dev).manual_seed(3)
        h = torch.randn((w.B, w.NH, w.S, w.DV), device=dev, generator=g)
        o = torch.randn(h.shape, device=dev, generator=g).to(torch.bfloat16)
        gam = torch.ones((w.NH, w.DV), device=dev)
        bet = torch.zeros((w.NH, w.DV), device=dev)
        y = torch.empty(h.shape, dtype=torch.bfloat16, device=dev)
        for _ in range(2):
            B.mlstm_groupnorm_gate(h, o, gam, bet, 1e-5, out=y)
    elif kind == "decode_multi":
        w = DEC
        T = 16
        g = torch.Generator(device=dev).manual_seed(0)
        C = torch.randn((w.B, w.NH, w.DV, w.DQK), device=dev, generator=g)
        n = torch.randn((w.B, w.NH, w.DQK), device=dev, generator=g)
        m = torch.zeros((w.B, w.NH), device=dev)
        q, k = (torch.randn((w.B, w.NH, T, w.DQK), device=dev, generator=g).to(torch.bfloat16) for _ in range(2))
        v = torch.randn((w.B, w.NH, T, w.DV), device=dev, generator=g).to(torch.bfloat16)
        ig, fg = (torch.randn((w.B, w.NH, T), device=dev, generator=g) for _ in range(2))
        for _ in range(2):
            B.mlstm_step_multi(q, k, v, ig, fg, C, n, m, h_dtype=torch.float32)
    else:
        w = DEC
        P = w.B * w.NH
        g = torch.Generator(device=dev).manual_seed(0)
        C = torch.randn((w.B, w.NH, w.DV, w.DQK), device=dev, generator=g)
        n = torch.randn((w.B, w.NH, w.DQK), device=dev, generator=g)
        m = torch.zeros((w.B, w.NH), device=dev)
        q, k = (torch.randn((w.B, w.NH, w.DQK), device=dev, generator=g).to(torch.bfloat16) for _ in range(2))
        v = torch.randn((w.B, w.NH, w.DV), device=dev, generator=g).to(torch.bfloat16)
        ig, fg = (torch.randn((w.B, w.NH), device=dev, generator=g) for _ in range(2))
        for _ in range(2):
            B.mlstm_step(q, k, v, ig, fg, C, n, m, h_dtype=torch.float32)
        del P
    torch.cuda.synchronize()
    print(f"profile {kind} done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["1p3b", "350m", "stress"], default="1p3b",
                    help="forward workload (default: the 1.3B-style layer)")
    ap.add_argument("--profile", choices=["fwd", "decode", "decode_multi", "gn", "bwd"], default=None,
                    help="run one small forward or decode step for ncu captures and exit")
    args = ap.parse_args()
    global FWD
    FWD = W.WORKLOADS[args.workload]
    if args.profile:
        run_profile(args.profile)
        return
    rank, local, world = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
