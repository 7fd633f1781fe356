#!/usr/bin/env python
"""Benchmark of the GGUF Q4_K/Q6_K x Q8 integer matmul path on GB300.

One step = one decode pass of the Llama-3-8B-shaped 32-layer sweep at M=8:
per layer, xq_layer_mixed quantizes the layer's four fp32 inputs to Q8 and
runs the seven Q4_K projections (Q, K, V, O, gate, up, down). All 3.93 GB of
weights stay resident in HBM (far larger than the 129 MB L2, so every step
streams them from HBM; no flush needed). The metric is weight GB/s: the
algorithmic weight bytes (144/256 B per Q4_K weight, 210/256 B per Q6_K
weight) per step over the step time.

Prints ONE JSON line (rank 0). Extra objects on it:
  by_m        the same sweep at M = 1, 2, 4, 8;
  roofline    the dominant kernel (the Q4_K matmul), bytes per launch over
              its CUDA-event launch time, against the measured HBM peak;
  secondary   the other workloads: Qwen2.5-1.5B and Qwen3-8B mixed layers
              (weights rotated over >= 3x L2 of copies) and the M=512
              Qwen3-8B FFN prefill tile;
  cpu_baseline the CPU oracle on a bounded sample of the same sweep;
  e2e         the same metric through the public API with pinned host
              inputs/outputs copied inside the timed region (the step's
              activations and outputs packed, one copy per direction).

`--impl reference` times the CPU oracle instead (rank 0 only).
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

from gguf_quant_integer_gb300 import synth  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
HEADLINE = "llama3-8b-32layer"


# The headline metric, the same string on both arms.
METRIC = "Q4_K/Q6_K x Q8 matmul weight GB/s (M=%d) and %% of GB300 HBM roofline"
# workloads --profile-workload runs (one launch per call)
PROFILE_WORKLOADS = ("prefill512-up", "prefill512-down", "prefill512-q8_0", "qwen3-q6k-layer", "q4km-q6k-layer",
                     "qwen3-layer", "llama3-layer", "iq4xs-ffn-up", "q8_0-qwen25-layer", "qwen25-layer")


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    # 200 steps of the headline sweep take about 0.25 s: enough clock samples
    # (every 20 ms) inside the timed region
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["xq", "reference"], default="xq")
    p.add_argument("--m", type=int, default=8, help="tokens per step (headline sweep)")
    p.add_argument("--no-secondary", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-sample-layers", type=int, default=8)
    p.add_argument("--layers", type=int, default=0,
                   help="run only the first L layers of the sweep (0 = all; small cases for ncu)")
    p.add_argument("--profile-workload", choices=sorted(PROFILE_WORKLOADS), default=None,
                   help="run one workload's launches (warmup + steps) without timing, for ncu captures")
    return p.parse_args(argv)


# ------------------------------------------------------------ multi-rank

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend: str):
    rank, world, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            os.environ.setdefault("MASTER_PORT", "29511")
            dist.init_process_group(backend, rank=rank, world_size=world)
    return rank, world


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int, device=None) -> float:
    """The slowest rank's value (timing is taken as the max over ranks)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(bytes_per_step_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job weight GB/s: every rank streams its own replica each step."""
    return bytes_per_step_per_rank * world / max_seconds / 1e9


# ------------------------------------------------------------ peaks, clocks

def measured_tensor_peak():
    """Dense fp16/bf16 tensor peak in TFLOP/s: the measured bf16 burst figure
    (fp16 runs at the bf16 rate), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                v = json.load(f).get("bf16_tflops")
            if v:
                return float(v), "measured"
        except Exception:
            pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            v = d.get("hbm_gbs") or d.get("hbm_GBps") or d.get("hbm")
            if isinstance(v, dict):
                v = v.get("value")
            if v:
                return float(v), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"xq_clocks_{os.getpid()}.csv")

    def start(self):
        """Start sampling and wait until the first sample is written, so the
        sampler is already running when the timed region begins."""
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def mark(self, name):
        setattr(self, name, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    sm.append(float(parts[2]))
                    smax.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[6:10]):
                    if v.lower() == "active":
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle

def oracle_sweep_seconds(wl, M, layers, host_weights, host_inputs, threads=1):
    """Time the CPU oracle over `layers` layers of the sweep (quantize the
    layer inputs, then every projection) with `threads` host threads sharing
    out output rows. Returns (seconds, weight bytes)."""
    import oracle
    oracle.build()
    oracle.set_threads(threads)
    nbytes = 0
    t0 = time.perf_counter()
    for l in layers:
        q8 = [oracle.quantize_q8(x) for x in host_inputs[l]]
        for t, p in enumerate(wl.projs):
            qs, d8, _ = q8[p.input]
            oracle.matmul(p.qtype, host_weights[l][t], qs, d8, p.K)
            nbytes += synth.weight_bytes(p.qtype, p.N, p.K)
    dt = time.perf_counter() - t0
    oracle.set_threads(1)
    return dt, nbytes


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    wl = synth.WORKLOADS[HEADLINE]
    M = args.m
    layers_per_step = 1
    sample = list(range(layers_per_step))
    host_w = {l: synth.gen_layer_weights(wl, l) for l in sample}
    host_x = {l: synth.gen_layer_inputs(wl, M, l) for l in sample}
    import oracle
    oracle.build()
    cores = oracle.set_threads(host_cores())
    for _ in range(args.warmup):
        oracle_sweep_seconds(wl, M, sample, host_w, host_x, threads=cores)
    secs, nbytes = [], 0
    for _ in range(args.steps):
        s, nbytes = oracle_sweep_seconds(wl, M, sample, host_w, host_x, threads=cores)
        secs.append(s)
    tot = sum(secs)
    value = nbytes * args.steps / tot / 1e9
    sample_desc = (f"layer 0 of the 32-layer sweep per step (Q8 quantize of its 4 inputs + 7 Q4_K "
                   f"projections, {nbytes / 1e6:.1f} MB of weights) at M={M}, output rows shared over "
                   f"{cores} host threads")
    line = {
        "impl": "reference", "metric": METRIC % M,
        "value": round(value, 6), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * tot / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded GGUF Q4_K blocks, fp32 N(0,1) activations)",
        "config": {"workload": HEADLINE, "M": M, "layers": wl.layers, "sample": sample_desc},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample_desc},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ GPU arm

def q6k_on_gemv(N, K):
    """Whether a Q6_K projection runs on the tensor-core GEMV (the rest run
    on the dp4a kernel): rows of 16-byte multiples, or N a multiple of 16
    times the count of consecutive rows whose bytes are (2, 4 or 8)."""
    row = (K // 256) * 210
    g = 1
    while g < 8 and (row * g) % 16:
        g *= 2
    return g == 1 or N % (16 * g) == 0


class Sweep:
    """All layers of a workload resident on the device, with per-M outputs."""

    def __init__(self, wl, layers_weights, device):
        import torch
        self.wl = wl
        self.device = device
        self.W = [[torch.from_numpy(w.reshape(-1)).to(device) for w in lw] for lw in layers_weights]
        self.n_inputs = 1 + max(p.input for p in wl.projs)
        self.state = {}

    def prepare(self, M, inputs_host):
        """Device inputs, outputs and workspace for batch M."""
        import torch
        from gguf_quant_integer_gb300 import xq
        ins = [[torch.from_numpy(x).to(self.device) for x in li] for li in inputs_host]
        ys = [[torch.empty((M, p.N), dtype=torch.float32, device=self.device) for p in self.wl.projs]
              for _ in self.W]
        descs = [[(p.qtype, p.N, p.K, self.W[l][t], ys[l][t], p.input) for t, p in enumerate(self.wl.projs)]
                 for l in range(len(self.W))]
        wsb = xq.layer_workspace_bytes(descs[0], self.n_inputs, M)
        ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=self.device)
        self.state[M] = (ins, ys, descs, ws)

    def step(self, M):
        from gguf_quant_integer_gb300 import xq
        ins, ys, descs, ws = self.state[M]
        for l in range(len(self.W)):
            xq.layer_mixed(descs[l], ins[l], M, ws)

    def launches_per_step(self, M):
        """Kernel launches of one step, following xq_layer_mixed's dispatch:
        one quantize launch per 8 inputs; for M <= 8 one grouped GEMV launch
        per weight type and 8 projections, plus one dp4a launch per Q6_K
        projection whose rows are not 16-byte multiples; for M > 8 one tile
        launch per projection."""
        used = len({p.input for p in self.wl.projs})
        per_layer = -(-used // 8)
        if M > 8:
            per_layer += len(self.wl.projs)
        else:
            grouped = {synth.Q4_K: 0, synth.Q6_K: 0}
            for p in self.wl.projs:
                if p.qtype == synth.Q4_K or q6k_on_gemv(p.N, p.K):
                    grouped[p.qtype] += 1
                else:
                    per_layer += 1
            per_layer += sum(-(-n // 8) for n in grouped.values())
        return len(self.W) * per_layer

    def bytes_per_step(self):
        return len(self.W) * self.wl.layer_weight_bytes()


def time_region(fn, steps, warmup, world, device):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def per_launch_matmul_times(sweep, M, reps=3):
    """CUDA-event duration of every projection launch of one sweep (the
    dominant kernel), on the stream the kernels run on. Returns a list of
    (qtype, bytes, seconds) per launch (average over reps sweeps)."""
    import torch
    from gguf_quant_integer_gb300 import xq
    ins, ys, descs, ws = sweep.state[M]
    s = torch.cuda.current_stream()
    wl = sweep.wl
    recs = []
    for _ in range(reps):
        evs = []
        for l in range(len(sweep.W)):
            bufs = {}
            for i in sorted({p.input for p in wl.projs}):
                bufs[i] = xq.quantize_q8(ins[l][i])
            for t, p in enumerate(wl.projs):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(s)
                xq.matmul(p.qtype, sweep.W[l][t], bufs[p.input], M, p.N, p.K, y=ys[l][t])
                b.record(s)
                evs.append((p, a, b))
        torch.cuda.synchronize()
        recs.append([(p.qtype, synth.weight_bytes(p.qtype, p.N, p.K), a.elapsed_time(b) / 1e3)
                     for p, a, b in evs])
    out = []
    for i in range(len(recs[0])):
        out.append((recs[0][i][0], recs[0][i][1], sum(r[i][2] for r in recs) / reps))
    return out


def per_layer_times(sweep, M, reps=3):
    """CUDA-event duration of every xq_layer_mixed call of one sweep, on the
    stream the kernels run on (its grouped Q4_K matmul launch plus the small
    grouped quantize launch before it). Returns seconds per layer, averaged
    over reps sweeps."""
    import torch
    from gguf_quant_integer_gb300 import xq
    ins, ys, descs, ws = sweep.state[M]
    s = torch.cuda.current_stream()
    tot = [0.0] * len(sweep.W)
    for _ in range(reps):
        evs = []
        for l in range(len(sweep.W)):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            xq.layer_mixed(descs[l], ins[l], M, ws)
            b.record(s)
            evs.append((a, b))
        torch.cuda.synchronize()
        for l, (a, b) in enumerate(evs):
            tot[l] += a.elapsed_time(b) / 1e3
    return [t / reps for t in tot]


def per_layer_gemv_times(sweep, M, reps=3):
    """CUDA-event duration of every layer's grouped matmul launch on its own
    (the dominant kernel), on the stream the kernels run on. Each layer gets
    its own workspace, which one xq_layer_mixed call fills with the layer's
    Q8 activations; then xq_debug_layer_matmuls re-runs just the matmul
    launch (one grouped launch for an all-Q4_K layer), layer after layer in
    sweep order, so every layer's weights were last read 31 layers (3.8 GB)
    earlier and stream from HBM. Returns seconds per layer, averaged over
    reps sweeps."""
    import torch
    from gguf_quant_integer_gb300 import xq
    ins, ys, descs, ws = sweep.state[M]
    wss = [torch.empty_like(ws) for _ in sweep.W]
    for l in range(len(sweep.W)):
        xq.layer_mixed(descs[l], ins[l], M, wss[l])
    s = torch.cuda.current_stream()
    tot = [0.0] * len(sweep.W)
    for _ in range(reps + 1):  # the first pass is a warm-up
        evs = []
        for l in range(len(sweep.W)):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            xq.debug_layer_matmuls(descs[l], sweep.n_inputs, M, wss[l])
            b.record(s)
            evs.append((a, b))
        torch.cuda.synchronize()
        if _ == 0:
            continue
        for l, (a, b) in enumerate(evs):
            tot[l] += a.elapsed_time(b) / 1e3
    return [t / reps for t in tot]


def gemv_back_to_back_time(sweep, M, steps, warmup, world, device):
    """Mean duration of one layer's grouped matmul launch when the launches
    run back to back as in the sweep: every layer gets its own workspace,
    which one xq_layer_mixed call fills with its Q8 activations, then the
    timed region runs xq_debug_layer_matmuls layer after layer, `steps`
    sweeps, CUDA events only at its ends (events between launches would
    break the programmatic-launch overlap the sweep runs with). Each layer's
    weights were last read 31 layers earlier and stream from HBM. Returns
    seconds per launch (one grouped launch per all-Q4_K layer)."""
    import torch
    from gguf_quant_integer_gb300 import xq
    ins, ys, descs, ws = sweep.state[M]
    wss = [torch.empty_like(ws) for _ in sweep.W]
    for l in range(len(sweep.W)):
        xq.layer_mixed(descs[l], ins[l], M, wss[l])

    def run():
        for l in range(len(sweep.W)):
            xq.debug_layer_matmuls(descs[l], sweep.n_inputs, M, wss[l])

    secs = time_region(run, steps, warmup, world, device)
    return max_over_ranks(secs, world, device) / (steps * len(sweep.W))


# Sources the grouped GEMV kernel is built from: a recorded ncu traffic
# figure stays valid only while their code is unchanged (comments and
# whitespace are not part of the hash).
GEMV_SOURCES = ("gemv_mma.cu", "xq_common.cuh", "xq_ptx.cuh")


def code_only(text: str) -> str:
    """C/C++ source with comments removed and whitespace runs collapsed
    (string literals are kept as they are)."""
    import re
    tok = re.compile(r'"(?:\\.|[^"\\])*"|/\*.*?\*/|//[^\n]*', re.S)
    out = tok.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", text)
    return " ".join(out.split())


def kernel_source_hash(names=GEMV_SOURCES, src=None) -> str:
    import hashlib
    src = src or os.path.join(ROOT, "gguf_quant_integer_gb300", "csrc")
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(src, name), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def read_ncu_traffic(kernel_key: str):
    """Per-launch DRAM bytes of `kernel_key` from the committed ncu summary,
    valid only if the hash of the kernel's sources recorded there matches the
    current one."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    digest = kernel_source_hash()
    with open(path) as f:
        for line in f:
            parts = line.strip().strip("|").split("|")
            parts = [p.strip() for p in parts]
            if len(parts) >= 4 and parts[0] == kernel_key and parts[3] == digest:
                try:
                    return float(parts[1]), parts[2]
                except ValueError:
                    return None
    return None


def gpu_arm(args):
    import torch
    rank, world = dist_init("nccl" if torch.cuda.is_available() else "gloo")
    _, _, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the xq path has no CPU fallback)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from gguf_quant_integer_gb300 import build, xq
    if rank == 0 or not os.path.exists(xq.LIB_PATH):
        build.build()
    barrier(world)
    xq.lib()

    wl = synth.WORKLOADS[HEADLINE]
    M = args.m
    n_layers = wl.layers if args.layers <= 0 else min(args.layers, wl.layers)
    host_w = [synth.gen_layer_weights(wl, l) for l in range(n_layers)]
    sweep = Sweep(wl, host_w, device)
    ms_list = sorted({1, 2, 4, 8, M})
    host_inputs = {m: [synth.gen_layer_inputs(wl, m, l) for l in range(n_layers)] for m in ms_list}
    for m in ms_list:
        sweep.prepare(m, host_inputs[m])
    nbytes = sweep.bytes_per_step()

    # ---- headline: timed region with clocks sampled during it
    clk = ClockSampler(local)
    clk.start()
    secs = time_region(lambda: sweep.step(M), args.steps, args.warmup, world, device)
    clocks = clk.stop()
    secs = max_over_ranks(secs, world, device)
    ms_per_step = 1e3 * secs / args.steps
    value = aggregate_value(nbytes, world, secs / args.steps)

    # ---- per-step distribution (context; outside the timed region): each of
    # 50 steps timed on its own with CUDA events
    import torch
    s_cur = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    for a, b in evs:
        a.record(s_cur)
        sweep.step(M)
        b.record(s_cur)
    torch.cuda.synchronize()
    per_step = sorted(a.elapsed_time(b) for a, b in evs)
    step_dist = {"n": len(per_step), "median_ms": round(statistics.median(per_step), 4),
                 "p10_ms": round(per_step[len(per_step) // 10], 4),
                 "p90_ms": round(per_step[(9 * len(per_step)) // 10], 4),
                 "note": "each step timed alone (events between steps), so adjacent layers of two steps do not overlap"}

    # ---- the same sweep at other M
    by_m = {}
    for m in ms_list:
        s = time_region(lambda: sweep.step(m), max(3, args.steps // 2), 3, world, device)
        s = max_over_ranks(s, world, device) / max(3, args.steps // 2)
        by_m[str(m)] = {"GBps": round(nbytes / s / 1e9, 1), "ms_per_step": round(1e3 * s, 4),
                        "tokens_per_s": round(m / s, 1)}

    # ---- dominant kernel: every layer's grouped Q4_K matmul launch (about
    # 90% of each layer's GPU time per the ncu launch list), timed alone and
    # back to back over a region; for context the same launches with events
    # around each, and the layer call with its quantize launch
    peak, peak_kind = measured_peaks()
    avg = gemv_back_to_back_time(sweep, M, args.steps, max(3, args.warmup), world, device)
    gts = per_layer_gemv_times(sweep, M)
    lts = per_layer_times(sweep, M)
    layer_bytes = wl.layer_weight_bytes()
    avg_each = sum(gts) / len(gts)
    avg_call = sum(lts) / len(lts)
    achieved = layer_bytes / avg / 1e9
    tr = read_ncu_traffic(f"gemv_mma_q4k_layer_M{M}")
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                "kernel": "gemv_mma_kernel<Q4_K>, the grouped launch of one layer, timed alone",
                "bytes_per_launch": layer_bytes, "avg_launch_us": round(1e6 * avg, 3),
                "avg_launch_note": "the 32 layers' grouped launches back to back (xq_debug_layer_matmuls, no quantize "
                                   "launches), CUDA events at the ends of the timed region, mean per launch",
                "avg_launch_us_events_each": round(1e6 * avg_each, 3),
                "layer_call_us": round(1e6 * avg_call, 3),
                "layer_call_note": "xq_layer_mixed per layer (quantize launch + GEMV launch), CUDA events per call",
                "traffic": (round(tr[0]) if tr else None),
                "traffic_note": (tr[1] if tr else "no ncu capture of the current kernel source")}
    # Context: every projection launched on its own (small projections get
    # small grids, so these are below the grouped figure).
    lt = per_launch_matmul_times(sweep, M, reps=1)
    per_proj = {}
    for t, p in enumerate(wl.projs):
        xs = lt[t::len(wl.projs)]
        bb = sum(b for _, b, _ in xs)
        tt = sum(s for _, _, s in xs)
        per_proj[p.name] = {"GBps": round(bb / tt / 1e9, 1), "us": round(1e6 * tt / len(xs), 2)}
    roofline["standalone_per_projection"] = per_proj

    # ---- e2e through the public API: pinned host in/out copied in the timed region
    e2e = None
    if not args.no_e2e:
        ins0, ys0, descs0, ws = sweep.state[M]
        # The step's activations live in one pinned host buffer and its
        # outputs in one device buffer, so each direction is one copy per
        # step (the layer calls read and write views into them).
        def pack(tensors, device_):
            sizes = [t.numel() for lt in tensors for t in lt]
            flat = torch.empty(sum(sizes), dtype=torch.float32, device=device_)
            views, o = [], 0
            for lt in tensors:
                row = []
                for t in lt:
                    row.append(flat[o:o + t.numel()].view(t.shape))
                    o += t.numel()
                views.append(row)
            return flat, views

        d_in, ins = pack(ins0, device)
        for li, l0 in zip(ins, ins0):
            for v, x in zip(li, l0):
                v.copy_(x)
        h_in = d_in.cpu().pin_memory()
        d_out, ys = pack(ys0, device)
        h_out = torch.empty(d_out.shape, dtype=torch.float32).pin_memory()
        descs = [[(t, n, k, w, ys[l][j], inp) for j, (t, n, k, w, _, inp) in enumerate(dl)]
                 for l, dl in enumerate(descs0)]
        h2d = h_in.numel() * 4
        d2h = h_out.numel() * 4

        # Copies overlap the layers: a copy stream brings the inputs over in
        # three chunks (layer 0, layers 1-3, the rest; at about 200 GB/s each
        # lands before its first layer starts) and takes the outputs back in
        # four (all but the last 8 layers, the next 6, then one and one), so
        # only layer 0's inputs and the last layer's outputs are exposed. A
        # wait on a copy ends the early start of the next launch, hence few
        # chunks.
        L = len(sweep.W)
        in_off = [0]
        for lt in ins0:
            in_off.append(in_off[-1] + sum(t.numel() for t in lt))
        out_off = [0]
        for lt in ys0:
            out_off.append(out_off[-1] + sum(t.numel() for t in lt))
        def spans(cuts):
            cuts = sorted({min(max(c, 0), L) for c in cuts} | {0, L})
            return [(a, b) for a, b in zip(cuts, cuts[1:]) if b > a]
        in_chunks = spans([1, 4])
        out_chunks = spans([L - 8, L - 2, L - 1])
        copy_s = torch.cuda.Stream(device)

        def e2e_step():
            cur = torch.cuda.current_stream()
            copy_s.wait_stream(cur)  # the previous step is done with d_in and d_out
            ev_in = []
            with torch.cuda.stream(copy_s):
                for a, b in in_chunks:
                    d_in[in_off[a]:in_off[b]].copy_(h_in[in_off[a]:in_off[b]], non_blocking=True)
                    ev_in.append(copy_s.record_event())
            ci = 0
            ev_out = []
            for l in range(L):
                if ci < len(in_chunks) and l == in_chunks[ci][0]:
                    cur.wait_event(ev_in[ci])
                    ci += 1
                xq.layer_mixed(descs[l], ins[l], M, ws)
                if any(l == b - 1 for _, b in out_chunks):
                    ev_out.append(cur.record_event())
            with torch.cuda.stream(copy_s):
                for (a, b), ev in zip(out_chunks, ev_out):
                    copy_s.wait_event(ev)
                    h_out[out_off[a]:out_off[b]].copy_(d_out[out_off[a]:out_off[b]], non_blocking=True)
            cur.wait_stream(copy_s)

        s = time_region(e2e_step, args.steps, max(3, args.warmup), world, device)
        s = max_over_ranks(s, world, device) / args.steps
        torch.cuda.synchronize()
        if not torch.equal(h_out, d_out.cpu()):  # every output chunk came back after its layers
            raise RuntimeError("e2e: host outputs differ from the device outputs")
        e2e = {"value": round(aggregate_value(nbytes, world, s), 1), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(1e3 * s, 4)}

    # ---- secondary workloads
    secondary = None
    if not args.no_secondary:
        secondary = secondary_workloads(device, world)

    # ---- CPU oracle on a bounded sample (rank 0, N=1 only)
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        import oracle
        oracle.build()
        S = max(1, min(args.cpu_sample_layers, n_layers))
        cores = oracle.set_threads(host_cores())
        # all host cores (output rows shared out), then one thread on a smaller sample
        cs, cb = oracle_sweep_seconds(wl, M, list(range(S)), host_w, host_inputs[M], threads=cores)
        S1 = max(1, min(2, n_layers))
        cs1, cb1 = oracle_sweep_seconds(wl, M, list(range(S1)), host_w, host_inputs[M], threads=1)
        cpu = {"value": round(cb / cs / 1e9, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "seconds": round(cs, 2),
               "sample": f"layers 0..{S - 1} of the 32-layer sweep at M={M} "
                         f"({cb / 1e9:.3f} GB of weights), C oracle with output rows shared over {cores} threads",
               "single_thread": {"value": round(cb1 / cs1 / 1e9, 5), "unit": "GB/s", "cores": 1,
                                 "seconds": round(cs1, 2),
                                 "sample": f"layers 0..{S1 - 1} ({cb1 / 1e9:.3f} GB of weights), one thread"}}

    if rank == 0:
        line = {
            "metric": METRIC % M,
            "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic (seeded GGUF Q4_K blocks, fp32 N(0,1) activations)",
            "config": {"workload": HEADLINE if n_layers == wl.layers else f"{HEADLINE} (first {n_layers} layers)",
                       "M": M, "layers": n_layers,
                       "weight_bytes_per_step": nbytes, "hidden": 4096, "ffn": 14336,
                       "l2": "weights 3.93 GB >> 129 MB L2, streamed from HBM every step; no flush",
                       "parallelism": f"replicas x{world}"},
            "hbm_frac": round(value / world / peak, 4), "hbm_peak_GBps": peak, "hbm_peak_source": peak_kind,
            "tokens_per_s": round(M * world / (secs / args.steps), 1),
            "gpu_launches": sweep.launches_per_step(M) * args.steps,
            "clocks": clocks, "roofline": roofline, "by_m": by_m, "step_distribution": step_dist,
            "e2e": e2e, "secondary": secondary, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    return 0


def secondary_workloads(device, world):
    """Single-layer workloads that fit in L2: weights rotated over enough
    device copies (>= 3x L2) that every launch reads from HBM."""
    import torch
    from gguf_quant_integer_gb300 import xq
    out = {}
    # the tiny Q4_K GEMV (256 x 2048, M = 1): quantize + matmul per call,
    # weights rotated over copies past 3x L2
    wl = synth.WORKLOADS["tiny-gemv"]
    p = wl.projs[0]
    w0 = torch.from_numpy(synth.gen_weight(p.qtype, wl.weight_seed(0, 0), p.N, p.K).reshape(-1)).to(device)
    wbytes = synth.weight_bytes(p.qtype, p.N, p.K)
    copies = max(3, -(-3 * L2_BYTES // wbytes))
    Ws = [w0] + [w0.clone() for _ in range(copies - 1)]
    x = torch.from_numpy(synth.gen_x(wl.x_seed(1), 1, p.K)).to(device)
    buf = xq.quantize_q8(x)
    y = torch.empty((1, p.N), dtype=torch.float32, device=device)

    def tiny_step():
        for c in range(copies):
            xq.quantize_q8(x, out=buf)
            xq.matmul(p.qtype, Ws[c], buf, 1, p.N, p.K, y=y)

    sec = max_over_ranks(time_region(tiny_step, 3, 2, world, device), world, device) / (3 * copies)
    out["tiny-gemv"] = {"M": 1, "N": p.N, "K": p.K, "rotated_copies": copies, "weight_bytes": wbytes,
                        "us_per_call": round(1e6 * sec, 3), "GBps": round(wbytes / sec / 1e9, 2),
                        "tokens_per_s": round(1 / sec, 1), "note": "quantize + matmul per call; launch-bound"}
    # the same calls replayed from CUDA graphs (slices of 172 calls, weights
    # still rotated): the GPU-side cost of a call without the host's launch
    # overhead, for context
    try:
        graphs = []
        for g0 in range(0, copies, 172):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for c in range(g0, min(copies, g0 + 172)):
                    xq.quantize_q8(x, out=buf)
                    xq.matmul(p.qtype, Ws[c], buf, 1, p.N, p.K, y=y)
            graphs.append(g)

        def graph_step():
            for g in graphs:
                g.replay()

        sg = max_over_ranks(time_region(graph_step, 3, 2, world, device), world, device) / (3 * copies)
        out["tiny-gemv"]["from_cuda_graph"] = {"us_per_call": round(1e6 * sg, 3), "GBps": round(wbytes / sg / 1e9, 2)}
        del graphs
    except Exception as e:  # capture is context, not the measurement
        out["tiny-gemv"]["from_cuda_graph"] = {"error": str(e)[:200]}
    # Q6_K rows that are not 16-byte multiples (the 8960 -> 1536 ffn_down of
    # the Qwen2.5-1.5B shape, 7350-byte rows): quantize + matmul per call
    N6, K6 = 1536, 8960
    wb6 = synth.weight_bytes(synth.Q6_K, N6, K6)
    copies = max(3, -(-3 * L2_BYTES // wb6))
    W6 = torch.from_numpy(synth.gen_q6k(61, N6, K6).reshape(-1)).to(device)
    W6s = [W6] + [W6.clone() for _ in range(copies - 1)]
    res6 = {}
    for M in (1, 8):
        x6 = torch.from_numpy(synth.gen_x(62 + M, M, K6)).to(device)
        buf6 = xq.quantize_q8(x6)
        y6 = torch.empty((M, N6), dtype=torch.float32, device=device)

        def q6_step():
            for c in range(copies):
                xq.quantize_q8(x6, out=buf6)
                xq.matmul(synth.Q6_K, W6s[c], buf6, M, N6, K6, y=y6)

        sec = max_over_ranks(time_region(q6_step, 5, 3, world, device), world, device) / (5 * copies)
        res6[str(M)] = {"us_per_call": round(1e6 * sec, 2), "GBps": round(wb6 / sec / 1e9, 1)}
    out["q6k-ffn_down-1536x8960"] = {"rotated_copies": copies, "weight_bytes": wb6, "by_m": res6,
                                     "path": "dp4a kernel (a single matmul of fewer than 128 row blocks; in a "
                                             "layer this projection runs on the tensor-core GEMV, split over K)",
                                     "note": "quantize + matmul per call"}
    for name in ("qwen2.5-1.5b-layer", "qwen2.5-1.5b-q4km-layer", "qwen3-8b-mixed-layer", "qwen2.5-1.5b-q8_0-layer"):
        wl = synth.WORKLOADS[name]
        lw = synth.gen_layer_weights(wl, 0)
        copies = max(3, -(-3 * L2_BYTES // wl.layer_weight_bytes()))
        base = [torch.from_numpy(w.reshape(-1)).to(device) for w in lw]
        reps = [base] + [[w.clone() for w in base] for _ in range(copies - 1)]
        res = {}
        for M in wl.ms:
            ins = [torch.from_numpy(x).to(device) for x in synth.gen_layer_inputs(wl, M, 0)]
            ys = [torch.empty((M, p.N), dtype=torch.float32, device=device) for p in wl.projs]
            descs = [[(p.qtype, p.N, p.K, reps[c][t], ys[t], p.input) for t, p in enumerate(wl.projs)]
                     for c in range(copies)]
            ws = torch.empty(max(256, xq.layer_workspace_bytes(descs[0], 4, M)), dtype=torch.uint8, device=device)

            def step():
                for c in range(copies):
                    xq.layer_mixed(descs[c], ins, M, ws)

            s = time_region(step, 5, 3, world, device)
            s = max_over_ranks(s, world, device) / (5 * copies)
            res[str(M)] = {"GBps": round(wl.layer_weight_bytes() / s / 1e9, 1), "us_per_layer": round(1e6 * s, 2),
                           "tokens_per_s": round(M / s, 1)}
            if wl.layer_weight_bytes() < L2_BYTES:
                # context only: the same layer repeated on one copy, its
                # weights resident in L2 ("hot")
                def hot():
                    for _ in range(copies):
                        xq.layer_mixed(descs[0], ins, M, ws)

                sh = max_over_ranks(time_region(hot, 5, 3, world, device), world, device) / (5 * copies)
                res[str(M)]["hot_l2_resident"] = {"GBps": round(wl.layer_weight_bytes() / sh / 1e9, 1),
                                                  "us_per_layer": round(1e6 * sh, 2)}
        out[name] = {"rotated_copies": copies, "layer_bytes": wl.layer_weight_bytes(), "by_m": res}
    # the Llama-3-8B-shaped layer with its down projection fed by
    # silu(gate) * up of the same call (xq_layer_mixed_ffn), against the same
    # layer with an independent down input (xq_layer_mixed)
    wl = synth.WORKLOADS["llama3-8b-32layer"]
    lw = synth.gen_layer_weights(wl, 0)
    copies = max(3, -(-3 * L2_BYTES // wl.layer_weight_bytes()))
    base = [torch.from_numpy(w.reshape(-1)).to(device) for w in lw]
    reps = [base] + [[w.clone() for w in base] for _ in range(copies - 1)]
    names = [p.name for p in wl.projs]
    gi, ui, di = names.index("gate"), names.index("up"), names.index("down")
    res = {}
    for M in (1, 8):
        ins = [torch.from_numpy(x).to(device) for x in synth.gen_layer_inputs(wl, M, 0)]
        ys = [torch.empty((M, p.N), dtype=torch.float32, device=device) for p in wl.projs]
        descs = [[(p.qtype, p.N, p.K, reps[c][t], ys[t], p.input) for t, p in enumerate(wl.projs)]
                 for c in range(copies)]
        ws = torch.empty(xq.layer_ffn_workspace_bytes(descs[0], 4, M, gi, ui, di), dtype=torch.uint8, device=device)
        ws2 = torch.empty(xq.layer_workspace_bytes(descs[0], 4, M), dtype=torch.uint8, device=device)
        row = {}
        for label, call in (("ffn_chain", lambda c: xq.layer_mixed_ffn(descs[c], gi, ui, di, ins[:3], M, ws)),
                            ("independent_down", lambda c: xq.layer_mixed(descs[c], ins, M, ws2))):
            def step(call=call):
                for c in range(copies):
                    call(c)
            sec = max_over_ranks(time_region(step, 5, 3, world, device), world, device) / (5 * copies)
            row[label] = {"us_per_layer": round(1e6 * sec, 2), "GBps": round(wl.layer_weight_bytes() / sec / 1e9, 1)}
        res[str(M)] = row
    out["llama3-8b-layer-swiglu-down"] = {"rotated_copies": copies, "layer_bytes": wl.layer_weight_bytes(),
                                          "by_m": res}
    # batched decode and prefill: the Qwen3-8B mixed layer at 16, 32 and 64
    # tokens (GEMV over 8-token chunks), 128, 256 and 512 (the tile kernel,
    # split over K where a projection's tiles leave SMs idle)
    wl = synth.WORKLOADS["qwen3-8b-mixed-layer"]
    lw = synth.gen_layer_weights(wl, 0)
    copies = max(3, -(-3 * L2_BYTES // wl.layer_weight_bytes()))
    base = [torch.from_numpy(w.reshape(-1)).to(device) for w in lw]
    reps = [base] + [[w.clone() for w in base] for _ in range(copies - 1)]
    res = {}
    for M in (16, 32, 64, 128, 256, 512):
        ins = [torch.from_numpy(x).to(device) for x in synth.gen_layer_inputs(wl, M, 0)]
        ys = [torch.empty((M, p.N), dtype=torch.float32, device=device) for p in wl.projs]
        descs = [[(p.qtype, p.N, p.K, reps[c][t], ys[t], p.input) for t, p in enumerate(wl.projs)]
                 for c in range(copies)]
        ws = torch.empty(max(256, xq.layer_workspace_bytes(descs[0], 4, M)), dtype=torch.uint8, device=device)

        def step():
            for c in range(copies):
                xq.layer_mixed(descs[c], ins, M, ws)

        sec = max_over_ranks(time_region(step, 3, 2, world, device), world, device) / (3 * copies)
        res[str(M)] = {"us_per_layer": round(1e6 * sec, 2), "GBps": round(wl.layer_weight_bytes() / sec / 1e9, 1),
                       "tokens_per_s": round(M / sec, 1)}
        if M > 64:
            flops = sum(2.0 * M * p.N * p.K for p in wl.projs)
            res[str(M)]["TOPS_int"] = round(flops / sec / 1e12, 1)
    out["qwen3-8b-mixed-layer-batched"] = {"rotated_copies": copies, "layer_bytes": wl.layer_weight_bytes(),
                                           "by_m": res,
                                           "path": "GEMV over 8-token chunks up to 64 tokens, tile above (K-split "
                                                   "where a projection has fewer 128x128 tiles than SMs)"}
    # IQ4_XS: the 17408 x 5120 ffn_up shape whose batch cost the IQ4_XS
    # entries of the Agent Telemetry log measure, with a synthetic codebook;
    # quantize + matmul per copy, weights rotated past L2
    N, K = 17408, 5120
    cb = synth.gen_codebook(0)
    w0 = torch.from_numpy(synth.gen_iq4xs(17, N, K).reshape(-1)).to(device)
    wbytes = synth.weight_bytes(synth.IQ4_XS, N, K)
    copies = max(3, -(-3 * L2_BYTES // wbytes))
    Ws = [w0] + [w0.clone() for _ in range(copies - 1)]
    res = {}
    for M in (1, 8):
        x = torch.from_numpy(synth.gen_x(18, M, K)).to(device)
        buf = xq.quantize_q8(x)
        y = torch.empty((M, N), dtype=torch.float32, device=device)

        def step():
            for c in range(copies):
                xq.quantize_q8(x, out=buf)
                xq.matmul_iq4xs_q8(Ws[c], cb, buf, M, N, K, y=y)

        sec = max_over_ranks(time_region(step, 5, 3, world, device), world, device) / (5 * copies)
        res[str(M)] = {"us": round(1e6 * sec, 2), "GBps": round(wbytes / sec / 1e9, 1)}
    # M > 8 on the tile kernel (the same quantize + matmul per copy)
    for M in (16, 64, 512):
        x = torch.from_numpy(synth.gen_x(19, M, K)).to(device)
        buf = xq.quantize_q8(x)
        y = torch.empty((M, N), dtype=torch.float32, device=device)

        def step():
            for c in range(copies):
                xq.quantize_q8(x, out=buf)
                xq.matmul_iq4xs_q8(Ws[c], cb, buf, M, N, K, y=y)

        sec = max_over_ranks(time_region(step, 3, 2, world, device), world, device) / (3 * copies)
        res[str(M)] = {"us": round(1e6 * sec, 2), "GBps": round(wbytes / sec / 1e9, 1),
                       "TOPS_int": round(2.0 * M * N * K / sec / 1e12, 1)}
    # Q8_0 on the tile kernel: the Qwen3-8B ffn_up shape (12288 x 4096) as Q8_0 at 512 tokens
    N, K, M = 12288, 4096, 512
    wq = torch.from_numpy(synth.gen_q8_0(23, N, K).reshape(-1)).to(device)
    x = torch.from_numpy(synth.gen_x(24, M, K)).to(device)
    bq = xq.quantize_q8(x)
    y = torch.empty((M, N), dtype=torch.float32, device=device)
    sec = max_over_ranks(time_region(lambda: xq.matmul(synth.Q8_0, wq, bq, M, N, K, y=y), 5, 3, world, device),
                         world, device) / 5
    out["q8_0-ffn_up-prefill512"] = {"ms": round(1e3 * sec, 4), "TOPS_int": round(2.0 * M * N * K / sec / 1e12, 1),
                                     "weight_bytes": synth.weight_bytes(synth.Q8_0, N, K)}
    out["iq4xs-ffn_up-17408x5120"] = {"rotated_copies": copies, "weight_bytes": wbytes, "by_m": res,
                                      "codebook": "synthetic (the pages do not print the format's table)"}
    # prefill tile M=512: up (Q4_K) then down (Q6_K), each launch timed on its own
    wl = synth.WORKLOADS["qwen3-8b-ffn-prefill512"]
    M = 512
    lw = synth.gen_layer_weights(wl, 0)
    Wd = [torch.from_numpy(w.reshape(-1)).to(device) for w in lw]
    # the chain the workload describes: x -> ffn_up -> y_up -> ffn_down
    x_up = torch.from_numpy(synth.gen_layer_inputs(wl, M, 0)[wl.projs[0].input]).to(device)
    ys = [torch.empty((M, p.N), dtype=torch.float32, device=device) for p in wl.projs]
    ins = [x_up, ys[0]]
    bufs = [xq.quantize_q8(x_up), xq.quantize_q8(ys[0])]
    launches = []
    for t, p in enumerate(wl.projs):
        launches.append((f"quantize_{p.name}", lambda t=t: xq.quantize_q8(ins[t], out=bufs[t]), 0.0))
        launches.append((p.name, lambda t=t, p=p: xq.matmul(p.qtype, Wd[t], bufs[t], M, p.N, p.K, y=ys[t]),
                         2.0 * M * p.N * p.K))
    reps = 10
    for _ in range(3):
        for _, fn, _ in launches:
            fn()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(launches) + 1)] for _ in range(reps)]
    for r in range(reps):
        for i, (_, fn, _) in enumerate(launches):
            ev[r][i].record()
            fn()
        ev[r][-1].record()
    torch.cuda.synchronize()
    per = {}
    for i, (name, _, flops) in enumerate(launches):
        ms = sorted(ev[r][i].elapsed_time(ev[r][i + 1]) for r in range(reps))[reps // 2]
        per[name] = {"ms": round(ms, 4)}
        if flops:
            per[name]["TOPS"] = round(flops / (ms * 1e-3) / 1e12, 1)
    total = sorted(ev[r][0].elapsed_time(ev[r][-1]) for r in range(reps))[reps // 2]
    flops = sum(2.0 * M * p.N * p.K for p in wl.projs)
    peak, peak_src = measured_tensor_peak()
    tops = flops / (total * 1e-3) / 1e12
    out[wl.key] = {"M": M, "ms": round(total, 4), "TOPS_int": round(tops, 1),
                   "tensor_frac": round(tops / peak, 4), "tensor_peak_TFLOPs": peak, "tensor_peak_source": peak_src,
                   "GBps_weights": round(wl.layer_weight_bytes() / (total * 1e-3) / 1e9, 1), "per_launch": per,
                   "path": "tcgen05 tile kernel: exact-integer fp16 operands, 32-block accumulators in TMEM",
                   "chain": "x -> Q8 -> ffn_up -> y_up -> Q8 -> ffn_down (down reads up's output)"}
    return out


def profile_workload(args):
    """Run the launches of one named workload `warmup + steps` times and exit.
    No timing: the process exists to be captured by ncu (one launch per call
    of the workload: one grouped layer GEMV, or one tile-kernel matmul)."""
    import torch
    from gguf_quant_integer_gb300 import xq
    device = torch.device("cuda")
    name = args.profile_workload
    if name in ("prefill512-up", "prefill512-down"):
        wl = synth.WORKLOADS["qwen3-8b-ffn-prefill512"]
        p = wl.projs[0 if name.endswith("up") else 1]
        t = wl.projs.index(p)
        M = args.m if args.m > 64 else 512  # the workload's 512 tokens unless --m gives a tile-sized count
        W = torch.from_numpy(synth.gen_layer_weights(wl, 0)[t].reshape(-1)).to(device)
        x = torch.from_numpy(synth.gen_layer_inputs(wl, M, 0)[p.input]).to(device)
        buf = xq.quantize_q8(x)
        y = torch.empty((M, p.N), dtype=torch.float32, device=device)
        run = lambda: xq.matmul(p.qtype, W, buf, M, p.N, p.K, y=y)
    elif name == "prefill512-q8_0":
        # the Qwen3-8B ffn_up shape (12288 x 4096) as Q8_0 on the tile kernel, as the bench's secondary line
        N, K = 12288, 4096
        M = args.m if args.m > 64 else 512
        W = torch.from_numpy(synth.gen_q8_0(23, N, K).reshape(-1)).to(device)
        buf = xq.quantize_q8(torch.from_numpy(synth.gen_x(24, M, K)).to(device))
        y = torch.empty((M, N), dtype=torch.float32, device=device)
        run = lambda: xq.matmul(synth.Q8_0, W, buf, M, N, K, y=y)
    elif name == "iq4xs-ffn-up":
        # IQ4_XS 17408 x 5120 (47.3 MB), synthetic codebook, M from --m
        N, K, M = 17408, 5120, args.m
        W = torch.from_numpy(synth.gen_iq4xs(17, N, K).reshape(-1)).to(device)
        cb = synth.gen_codebook(0)
        buf = xq.quantize_q8(torch.from_numpy(synth.gen_x(18, M, K)).to(device))
        y = torch.empty((M, N), dtype=torch.float32, device=device)
        run = lambda: xq.matmul_iq4xs_q8(W, cb, buf, M, N, K, y=y)
    else:
        wl = synth.WORKLOADS[{"qwen3-q6k-layer": "qwen3-8b-mixed-layer", "q4km-q6k-layer": "qwen2.5-1.5b-q4km-layer",
                              "qwen3-layer": "qwen3-8b-mixed-layer",
                              "qwen25-layer": "qwen2.5-1.5b-layer",
                              "q8_0-qwen25-layer": "qwen2.5-1.5b-q8_0-layer"}.get(name, "llama3-8b-32layer")]
        # the *-q6k-layer workloads keep only the layer's Q6_K projections
        q6_only = name.endswith("q6k-layer")
        keep = [t for t, p in enumerate(wl.projs) if not q6_only or p.qtype == synth.Q6_K]
        M = args.m
        weights = synth.gen_layer_weights(wl, 0)
        inputs = synth.gen_layer_inputs(wl, M, 0)
        projs = [wl.projs[t] for t in keep]
        used = sorted({p.input for p in projs})
        remap = {i: k for k, i in enumerate(used)}
        Wd = [torch.from_numpy(weights[t].reshape(-1)).to(device) for t in keep]
        xs = [torch.from_numpy(inputs[i]).to(device) for i in used]
        ys = [torch.empty((M, p.N), dtype=torch.float32, device=device) for p in projs]
        desc = [(p.qtype, p.N, p.K, Wd[k], ys[k], remap[p.input]) for k, p in enumerate(projs)]
        ws = torch.empty(xq.layer_workspace_bytes(desc, len(xs), M), dtype=torch.uint8, device=device)
        run = lambda: xq.layer_mixed(desc, xs, M, ws)
    for _ in range(args.warmup + args.steps):
        run()
    torch.cuda.synchronize()
    print(f"profile workload {name}: {args.warmup + args.steps} calls done", flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return reference_arm(args)
    if args.profile_workload:
        return profile_workload(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
