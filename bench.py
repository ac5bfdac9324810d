"""Benchmark of the 8-bit rollout linear-layer hot path on GB300.

Headline (one JSON line on rank 0): the per-step requant of a whole
Qwen2.5-32B-shaped model plus its prefill GEMMs.  One step is one pass of the
hot path over that model:
  A1  requant all 64 layers x {qkv 5120->7168, o_proj 5120->5120, gate_up
      5120->55296, down 27648->5120} (256 bf16 tensors, 31.2 G values, one
      grouped launch) into 128x128-block E4M3 codes + fp32 scales; every weight
      went through a policy update W <- bf16(W + N(0, 1e-4)) first (set-up,
      untimed);
  A2  quantize the four prefill inputs X [8192, K] into 1x128-group E4M3;
  A3  run the four block-scaled FP8 GEMMs at M = 8192 on the codes of layer
      s % 64 (written by this step's requant) -> bf16 Y [8192, N].
value = algorithmic bytes of the step / step time (GB/s).  The model's 62.4 GB
of weights and 31.2 GB of codes are far above L2, so every step streams them
from HBM.  CUDA events around every part inside the timed region give each
kernel's time, from which the line's roofline list is built: the requant on
HBM, the prefill GEMMs on the FP8 tensor pipe, and the decode GEMMs of the
32B decode sweep (M in {1, 8, 32, 128, 256}, graphs over > 3x L2 of weight
copies) on HBM.

Other rows are measured as sub-benchmarks under "extras" (not in `value`):
the Qwen2.5-7B decode step at M = 64, prefill-size activation quant, the
grouped MoE GEMM, the FP8-vs-INT8 rollout mismatch KL, the FP8 KV-cache
quant, the TIS/MIS weights and the INT8 W8A8 path.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--extras all|none]
    python bench.py --impl reference ...     # the CPU oracle on a bounded sample
Under torchrun each rank is an independent replica (the path does not shard).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from precision_rl_rollout_gb300 import synth  # noqa: E402

METRIC = "FP8 W8A8 GEMM TFLOP/s (prefill), HBM GB/s (decode M<=256), requant GB/s"
UNIT = "GB/s"
DECODE_M = 64
COPIES = 4
L2_BYTES = 129 * 2 ** 20
LAYERS = synth.QWEN25_32B_LAYERS
PREFILL_M = synth.PREFILL_M

# ncu-measured DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per
# launch of each roofline kernel, valid only for the source it was taken on
# (checked by hash; null otherwise), from the committed profile summaries.
#  - requant: one Qwen2.5-32B layer (4 tensors, 487.6 M values) per launch,
#    scaled to the 64-layer launch by the values processed;
#  - prefill: the four M = 8192 GEMMs of the 32B layer, summed;
#  - decode: one launch of the worst decode-sweep shape.
NCU_TRAFFIC = {"kernel": "quant_weight_block_kernel", "source_sha1": "14ed2e9e98c2a88ac5aaac25907debfb6bbd1bf2",
               "bytes_per_value": (1950416128 + 918452736) / (2 * sum(s.elems for s in synth.QWEN25_32B)),
               "profile": "profiles/requant_weight_block_qwen32b_2layers.md"}
NCU_TRAFFIC_PREFILL = {"kernel": "gemm_fp8_prefill_kernel", "source_sha1": "a0a012e74cd88f9bda36e610f17a2232643fb487",
                       "bytes_per_step": (107077888 + 89341184) + (88692736 + 53771520) + (1350391296 + 879037440)
                       + (2134614528 + 78475776),
                       "profile": "profiles/prefill_gemm_qwen32b_m8192_four_shapes.md"}
NCU_TRAFFIC_DECODE = {"kernel": "FP8 GEMM at a decode size", "source_sha1": "45b109e770ec644a2e355791db05740407eaebce",
                      "case": "o_proj_M256", "bytes_per_launch": 27614208 + 15736832,
                      "profile": "profiles/decode_gemm_qwen32b_o_proj_m256.md"}


# ------------------------------------------------------------------ algorithmic bytes

def requant_bytes(N, K):
    """bf16 read + e4m3 write + one fp32 scale per 128x128 block."""
    return 2 * N * K + N * K + 4 * (N // 128) * (K // 128)


def act_quant_bytes(M, K):
    return 2 * M * K + M * K + 4 * M * (K // 128)


def gemm_bytes(M, N, K):
    """e4m3 W + its scales + e4m3 X + its scales + bf16 Y."""
    return N * K + 4 * (N // 128) * (K // 128) + M * K + 4 * M * (K // 128) + 2 * M * N


def int8_gemm_bytes(M, N, K):
    return N * K + 4 * N + M * K + 4 * M + 2 * M * N


def step_bytes(shapes, M):
    """The Qwen2.5-7B decode step: requant + act quant + GEMM of each layer."""
    return sum(requant_bytes(s.N, s.K) + act_quant_bytes(M, s.K) + gemm_bytes(M, s.N, s.K)
               for s in shapes)


def model_step_parts(shapes=synth.QWEN25_32B, layers=LAYERS, M=PREFILL_M):
    """Algorithmic bytes (and GEMM FLOPs) of the headline step: the requant of
    `layers` copies of `shapes`, the act quant of one [M, K] input per shape and
    one [M, K] x [N, K]^T GEMM per shape."""
    return {"requant_bytes": layers * sum(requant_bytes(s.N, s.K) for s in shapes),
            "act_quant_bytes": sum(act_quant_bytes(M, s.K) for s in shapes),
            "gemm_bytes": sum(gemm_bytes(M, s.N, s.K) for s in shapes),
            "gemm_flops": sum(2 * M * s.N * s.K for s in shapes)}


def model_step_bytes(**kw):
    p = model_step_parts(**kw)
    return p["requant_bytes"] + p["act_quant_bytes"] + p["gemm_bytes"]


def fp8_peak_tflops(peaks):
    """Dense FP8 tensor peak: the measured bf16 cuBLAS rate x 2 (the nominal
    FP8 : BF16 dense ratio, 4.5 : 2.25 PFLOP/s)."""
    return 2.0 * peaks["bf16_tflops"], 2.0 * peaks["bf16_tflops_sustained"]


# ------------------------------------------------------------------ environment

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _smi_id(device: int) -> str:
    """nvidia-smi addresses GPUs by PCI bus id; torch's index is relative to
    CUDA_VISIBLE_DEVICES, so translate through the PCI location."""
    try:
        p = torch.cuda.get_device_properties(device)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return str(device)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value over all ranks (the slowest replica sets the time)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while the
    timed region runs, written to a CSV in a temporary directory (or `path`)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int, rank: int = 0, path: str | None = None):
        self.smi_id = _smi_id(device)
        self.proc = None
        self.path = path or os.path.join(tempfile.gettempdir(), f"fp8rl_bench_clocks_{os.getpid()}_rank{rank}.csv")

    def __enter__(self):
        try:
            d = os.path.dirname(self.path)
            if d:
                os.makedirs(d, exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.smi_id}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        return summarize_clocks(open(self.path).read().splitlines())


def summarize_clocks(lines):
    """Median SM clock, the maximum, and the throttle reasons seen active."""
    sm, mx, reasons = [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            mx = float(f[2])
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def capture_graph(fn):
    """Capture fn's launches (library calls on the current stream) into a CUDA graph."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _flush_l2(buf):
    buf.add_(1)


def _time_op(fn, reps, flush=None, warm=3):
    """Median time of single launches (for ms-scale kernels), L2 flushed before each."""
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def _time_graph(calls, reps=10):
    """Per-call device time of `calls` (a list of no-arg library calls) captured
    back to back in one CUDA graph and replayed `reps` times."""
    for c in calls:
        c()
    torch.cuda.synchronize()
    g = capture_graph(lambda: [c() for c in calls])
    g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) / (reps * len(calls))


def _copies_for(nbytes):
    """Distinct weight copies so that one pass over them exceeds 3x L2."""
    return max(2, -(-3 * L2_BYTES // max(1, nbytes)))


# ------------------------------------------------------------------ headline: 32B requant + prefill

class Model32B:
    """A Qwen2.5-32B-shaped model on the device: 64 layers x 4 bf16 weights
    (after one policy update), their E4M3 codes and block scales, and the four
    prefill inputs X [8192, K] with their codes and the outputs Y [8192, N]."""

    def __init__(self, fb, dev, layers=LAYERS, M=PREFILL_M):
        self.shapes = synth.QWEN25_32B
        self.layers, self.M = layers, M
        self.W, self.Wq, self.Ws = [], [], []
        for layer in range(layers):
            for i, s in enumerate(self.shapes):
                seed = synth.seed_for(4, 0) + 1000 * layer + i
                W = synth.weight_bf16_direct(s.N, s.K, seed, device=dev)
                synth.policy_update_(W, seed + 500)                        # A0, untimed
                self.W.append(W)
                self.Wq.append(torch.empty(s.N, s.K, dtype=torch.uint8, device=dev))
                self.Ws.append(torch.empty(s.N // 128, s.K // 128, dtype=torch.float32, device=dev))
        self.requant = fb.GroupedRequant(list(zip(self.W, self.Wq, self.Ws)))
        self.X = [synth.activation(M, s.K, synth.seed_for(4, 1) + i, device=dev) for i, s in enumerate(self.shapes)]
        self.Xq = [torch.empty(M, s.K, dtype=torch.uint8, device=dev) for s in self.shapes]
        self.Xs = [torch.empty(s.K // 128, M, dtype=torch.float32, device=dev) for s in self.shapes]
        self.Y = [torch.empty(M, s.N, dtype=torch.bfloat16, device=dev) for s in self.shapes]
        self.ws = [torch.empty(max(16, fb.fp8rl_gemm_workspace_bytes(M, s.N, s.K)), dtype=torch.uint8, device=dev)
                   for s in self.shapes]

    def codes(self, layer, i):
        j = layer * len(self.shapes) + i
        return self.Wq[j], self.Ws[j]

    def act_quant(self, fb, i):
        fb.fp8rl_quant_act_group(self.X[i], self.Xq[i], self.Xs[i])

    def gemm(self, fb, layer, i):
        Wq, Ws = self.codes(layer, i)
        fb.fp8rl_gemm_w8a8_block(self.Xq[i], self.Xs[i], Wq, Ws, Y=self.Y[i], workspace=self.ws[i])


def time_headline(fb, args, dev, world, rank, model):
    """K timed steps (requant of the whole model, act quant of the four prefill
    inputs, the four prefill GEMMs on layer s % 64), bracketed by barrier +
    synchronize, with CUDA events on the launching stream between the parts of
    every step: the step time, and each roofline kernel's mean launch time over
    the timed region."""
    ns = len(model.shapes)
    stream = torch.cuda.current_stream()
    launches = 1 + ns + sum(fb.fp8rl_gemm_kernel_count(model.M, s.N, s.K, model.ws[i].numel())
                            for i, s in enumerate(model.shapes))

    def step(s, ev=None):
        layer = s % model.layers
        if ev is not None:
            ev[0].record(stream)
        model.requant()
        if ev is not None:
            ev[1].record(stream)
        for i in range(ns):
            model.act_quant(fb, i)
        if ev is not None:
            ev[2].record(stream)
        for i in range(ns):
            model.gemm(fb, layer, i)
            if ev is not None:
                ev[3 + i].record(stream)

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3 + ns)] for _ in range(args.steps)]
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device(), rank, args.clocks_out) as clk:
        for s in range(args.steps):
            step(args.warmup + s, evs[s])
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    total_ms = max_over_ranks(evs[0][0].elapsed_time(t1), world, dev)
    req_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    aq_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    gemm_ms = [statistics.mean(e[2 + i].elapsed_time(e[3 + i]) for e in evs) for i in range(ns)]
    step_ms = [e[0].elapsed_time(e[2 + ns]) for e in evs]
    assert fb.fp8rl_check_device_error() == 0
    return {"total_ms": total_ms, "req_ms": req_ms, "aq_ms": aq_ms, "gemm_ms": gemm_ms,
            "step_ms_pct": step_percentiles(step_ms), "clocks": clk.summary(), "launches_per_step": launches}


def step_percentiles(ms):
    """p10 / median / p90 of per-step times (linear interpolation between order statistics)."""
    xs = sorted(ms)
    if not xs:
        return None

    def q(f):
        pos = f * (len(xs) - 1)
        lo = int(pos)
        hi = min(lo + 1, len(xs) - 1)
        return xs[lo] + (xs[hi] - xs[lo]) * (pos - lo)
    return {"p10": q(0.1), "p50": q(0.5), "p90": q(0.9), "n": len(xs)}


def time_e2e(fb, args, dev, model, chunk_layers=8):
    """The same step through the public API from pinned host memory, the way an
    engine receiving a new policy would run it: every step copies all 64
    layers' bf16 weights host -> device (from one pinned host buffer per shape,
    reused for every layer) and the four prefill inputs, requantizes each chunk
    of 8 layers as soon as its copies have landed, runs act quant and the four
    prefill GEMMs, and reads the four Y back to pinned host memory.  Copies in,
    compute and copies out run on three streams, ordered by events, so the
    copies of the next chunk overlap the requant of this one."""
    shapes, ns = model.shapes, len(model.shapes)
    hW = [torch.empty(s.N, s.K, dtype=torch.bfloat16).pin_memory() for s in shapes]
    for i in range(ns):
        hW[i].copy_(model.W[i])                       # layer 0's weights as the host copy
    hX = [x.cpu().pin_memory() for x in model.X]
    hY = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in model.Y]
    chunks = [list(range(c, min(model.layers, c + chunk_layers))) for c in range(0, model.layers, chunk_layers)]
    req = [fb.GroupedRequant([(model.W[l * ns + i], model.Wq[l * ns + i], model.Ws[l * ns + i])
                              for l in ch for i in range(ns)]) for ch in chunks]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in chunks]       # chunk c's weights have landed
    ev_used = [torch.cuda.Event() for _ in chunks]     # chunk c's bf16 weights consumed by its requant
    ev_x, ev_done, ev_out = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
    for e in ev_used + [ev_done, ev_out]:              # every event recorded once before first use
        e.record(comp)
    h2d = model.layers * sum(t.numel() * t.element_size() for t in hW) + \
        sum(t.numel() * t.element_size() for t in hX)
    d2h = sum(t.numel() * t.element_size() for t in hY)

    def step(n):
        layer = n % model.layers
        for c, ch in enumerate(chunks):
            s_in.wait_event(ev_used[c])
            with torch.cuda.stream(s_in):
                for l in ch:
                    for i in range(ns):
                        model.W[l * ns + i].copy_(hW[i], non_blocking=True)
            ev_in[c].record(s_in)
        s_in.wait_event(ev_done)                       # the previous step's act quant has read X
        with torch.cuda.stream(s_in):
            for i in range(ns):
                model.X[i].copy_(hX[i], non_blocking=True)
        ev_x.record(s_in)
        for c in range(len(chunks)):
            comp.wait_event(ev_in[c])
            req[c]()
            ev_used[c].record(comp)
        comp.wait_event(ev_x)
        comp.wait_event(ev_out)                        # the previous step's Y has been read back
        for i in range(ns):
            model.act_quant(fb, i)
        for i in range(ns):
            model.gemm(fb, layer, i)
        ev_done.record(comp)
        s_out.wait_event(ev_done)
        with torch.cuda.stream(s_out):
            for i in range(ns):
                hY[i].copy_(model.Y[i], non_blocking=True)
        ev_out.record(s_out)

    steps = max(3, min(args.steps, 5))
    for n in range(3):
        step(n)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for n in range(steps):
        step(n)
    b.record(s_out)                    # the last read-back waits for the last compute and its copies in
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    assert fb.fp8rl_check_device_error() == 0
    del req
    return {"value": model_step_bytes() / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "host_link_gbs": (h2d + d2h) / (ms * 1e-3) / 1e9,
            "method": "64 layers' bf16 weights + 4 prefill inputs copied in per step (chunks of 8 layers, "
                      "requant of a chunk overlapping the next chunk's copies), act quant, 4 prefill GEMMs, "
                      "4 Y read back; copies in / compute / copies out on three streams"}


def decode_sweep_32b(fb, dev, reps=10):
    """A2 + A4 on the Qwen2.5-32B shapes at M in {1, 8, 32, 128, 256}: each GEMM
    walks distinct weight copies (> 3x L2) back to back in one CUDA graph.  No
    kernel in the graph writes weights, so the GEMMs pass
    FP8RL_GEMM_WEIGHTS_STABLE."""
    dec = {}
    for s in synth.QWEN25_32B:
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(3, 0), device=dev)
        Wq, Ws = fb.fp8rl_quant_weight_block(W)
        del W
        nc = _copies_for(s.N * s.K)
        Wqs = [Wq] + [Wq.clone() for _ in range(nc - 1)]
        Wss = [Ws] + [Ws.clone() for _ in range(nc - 1)]
        for M in synth.DECODE_M_SWEEP:
            X = synth.activation(M, s.K, synth.seed_for(3, 1), device=dev)
            Xq, Xs = fb.fp8rl_quant_act_group(X)
            Y = torch.empty(M, s.N, dtype=torch.bfloat16, device=dev)
            gws = torch.empty(max(16, fb.fp8rl_gemm_workspace_bytes(M, s.N, s.K)), dtype=torch.uint8, device=dev)
            ms = _time_graph([lambda c=c: fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wqs[c], Wss[c], Y=Y, workspace=gws,
                                                                   weights_stable=True)
                              for c in range(nc)], reps)
            aq = _time_graph([lambda: fb.fp8rl_quant_act_group(X, Xq, Xs)] * 16, reps)
            dec[f"{s.name}_M{M}"] = {"shape": s.name, "M": M, "N": s.N, "K": s.K,
                                     "gemm_us": ms * 1e3, "gemm_bytes": gemm_bytes(M, s.N, s.K),
                                     "gemm_gbs": gemm_bytes(M, s.N, s.K) / (ms * 1e-3) / 1e9,
                                     "gemm_tflops": 2 * M * s.N * s.K / (ms * 1e-3) / 1e12,
                                     "act_quant_us": aq * 1e3, "weight_copies": nc}
            del X, Xq, Xs, Y, gws
        del Wq, Ws, Wqs, Wss
    torch.cuda.empty_cache()
    assert fb.fp8rl_check_device_error() == 0
    return dec


# ------------------------------------------------------------------ roofline entries

def _file_sha1(*names):
    h = hashlib.sha1()
    for n in names:
        with open(os.path.join(ROOT, "precision_rl_rollout_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def requant_source_sha1(quant_cu=None, common_cuh=None):
    """sha1 of the requant kernel's own source: quant.cu up to its activation
    section (the file header, includes and the weight section) and common.cuh.
    The other quantizers in the file do not change it.  Texts (bytes) may be
    passed in; by default they are read from the tree."""
    csrc = os.path.join(ROOT, "precision_rl_rollout_gb300", "csrc")
    text = quant_cu if quant_cu is not None else open(os.path.join(csrc, "quant.cu"), "rb").read()
    common = common_cuh if common_cuh is not None else open(os.path.join(csrc, "common.cuh"), "rb").read()
    head = text.index(b"// ---------------------------------------------------------------- FP8 weights")
    tail = text.index(b"// ---------------------------------------------------------------- FP8 activations")
    if not head < tail:
        raise ValueError("quant.cu: the weight section must precede the activation section")
    return hashlib.sha1(text[:tail] + common).hexdigest()


def prefill_source_sha1():
    return _file_sha1("gemm_fp8_prefill.cu", "sm100_ptx.cuh", "common.cuh")


def decode_source_sha1():
    """Both GEMM kernels: the dispatch may give a decode size to either."""
    return _file_sha1("gemm_fp8_tc.cu", "gemm_fp8_prefill.cu", "sm100_ptx.cuh", "common.cuh")


def traffic_or_null(values=None):
    """ncu DRAM traffic of the requant launch over `values` bf16 values (the
    recorded bytes per value times the values), or None when the recorded
    figure was taken on other source."""
    if NCU_TRAFFIC["source_sha1"] != requant_source_sha1() or not NCU_TRAFFIC["bytes_per_value"]:
        return None
    if values is None:
        values = LAYERS * sum(s.elems for s in synth.QWEN25_32B)
    return NCU_TRAFFIC["bytes_per_value"] * values


def prefill_traffic_or_null():
    t = NCU_TRAFFIC_PREFILL
    return t["bytes_per_step"] if t["source_sha1"] and t["source_sha1"] == prefill_source_sha1() else None


def decode_traffic_or_null(case):
    t = NCU_TRAFFIC_DECODE
    ok = t["source_sha1"] and t["source_sha1"] == decode_source_sha1() and t["case"] == case
    return t["bytes_per_launch"] if ok else None


def roofline_entries(head, dec, peaks):
    """One entry per part of the metric: the requant (HBM) and the prefill GEMMs
    (FP8 tensor pipe) from the headline's timed region, and the decode GEMMs
    (HBM) of the 32B decode sweep at the M whose aggregate fraction is lowest."""
    parts = model_step_parts()
    hbm = peaks["hbm_gbs"]
    fp8, fp8_sus = fp8_peak_tflops(peaks)
    req_gbs = parts["requant_bytes"] / (head["req_ms"] * 1e-3) / 1e9
    ent = [{"part": "requant (A1)", "bound": "hbm", "kernel": "quant_weight_block_kernel (one grouped launch, "
            "64 layers x 4 Qwen2.5-32B weights)", "achieved": req_gbs, "peak": hbm, "unit": "GB/s",
            "frac": req_gbs / hbm, "traffic": traffic_or_null(),
            "algorithmic_bytes_per_launch": parts["requant_bytes"], "launch_ms": head["req_ms"],
            "peak_source": f"{peaks['source']} hbm_gbs (STREAM-style copy)", "config": "32B full-model requant"}]
    gemm_s = sum(head["gemm_ms"]) * 1e-3
    tfl = parts["gemm_flops"] / gemm_s / 1e12
    per_shape = {s.name: {"ms": head["gemm_ms"][i],
                          "tflops": 2 * PREFILL_M * s.N * s.K / (head["gemm_ms"][i] * 1e-3) / 1e12,
                          "frac": 2 * PREFILL_M * s.N * s.K / (head["gemm_ms"][i] * 1e-3) / 1e12 / fp8}
                 for i, s in enumerate(synth.QWEN25_32B)}
    ent.append({"part": "prefill GEMM (A3)", "bound": "tensor",
                "kernel": "gemm_fp8_prefill_kernel (4 launches: qkv, o_proj, gate_up, down at M=8192)",
                "achieved": tfl, "peak": fp8, "unit": "TFLOP/s", "frac": tfl / fp8, "frac_of_sustained": tfl / fp8_sus,
                "traffic": prefill_traffic_or_null(), "algorithmic_flops": parts["gemm_flops"],
                "algorithmic_bytes": parts["gemm_bytes"], "per_shape": per_shape,
                "peak_source": f"2 x {peaks['source']} bf16 cuBLAS burst (nominal FP8:BF16 dense = 2); "
                               f"frac_of_sustained uses 2 x the sustained bf16 figure",
                "config": "32B prefill, M=8192"})
    by_m = {}
    for r in dec.values():
        a = by_m.setdefault(r["M"], {"bytes": 0, "us": 0.0, "shapes": {}})
        a["bytes"] += r["gemm_bytes"]
        a["us"] += r["gemm_us"]
        a["shapes"][r["shape"]] = r["gemm_gbs"] / hbm
    worst_m = min(by_m, key=lambda m: by_m[m]["bytes"] / by_m[m]["us"])
    w = by_m[worst_m]
    gbs = w["bytes"] / (w["us"] * 1e-6) / 1e9
    worst_shape = min(w["shapes"], key=w["shapes"].get)
    ent.append({"part": "decode GEMM (A4)", "bound": "hbm",
                "kernel": f"the FP8 GEMM kernels the dispatch picks at decode sizes (gemm_fp8_decode_kernel, or "
                          f"gemm_fp8_prefill_kernel where its cost model is lower; each with its split-K "
                          f"reduction launch where planned), Qwen2.5-32B shapes at M={worst_m}, the sweep M with "
                          f"the lowest aggregate fraction",
                "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                "traffic": decode_traffic_or_null(f"{worst_shape}_M{worst_m}"),
                "algorithmic_bytes": w["bytes"], "per_shape_frac": w["shapes"],
                "frac_by_m": {str(m): (v["bytes"] / (v["us"] * 1e-6) / 1e9) / hbm for m, v in sorted(by_m.items())},
                "peak_source": f"{peaks['source']} hbm_gbs (STREAM-style copy)",
                "config": "32B decode sweep M in {1,8,32,128,256}, graphs over > 3x L2 of weight copies"})
    return ent


# ------------------------------------------------------------------ extra: the 7B decode step

class LayerSet:
    """One copy of the Qwen2.5-7B FP8 layer set: bf16 weights, their E4M3 codes
    and scales, the four layer inputs and their quantized forms, and the outputs."""

    def __init__(self, shapes, M, seed_base, dev):
        self.shapes = shapes
        self.W, self.Wq, self.Ws, self.X, self.Xq, self.Xs, self.Y = [], [], [], [], [], [], []
        for i, s in enumerate(shapes):
            W = synth.weight_bf16_direct(s.N, s.K, seed_base + 10 * i, device=dev)
            synth.policy_update_(W, seed_base + 10 * i + 5)           # A0, untimed
            self.W.append(W)
            self.Wq.append(torch.empty(s.N, s.K, dtype=torch.uint8, device=dev))
            self.Ws.append(torch.empty(s.N // 128, s.K // 128, dtype=torch.float32, device=dev))
            self.X.append(synth.activation(M, s.K, seed_base + 10 * i + 1, device=dev))
            self.Xq.append(torch.empty(M, s.K, dtype=torch.uint8, device=dev))
            self.Xs.append(torch.empty(s.K // 128, M, dtype=torch.float32, device=dev))
            self.Y.append(torch.empty(M, s.N, dtype=torch.bfloat16, device=dev))
        self.group = list(zip(self.W, self.Wq, self.Ws))


def run_requant(fb, ls):
    fb.fp8rl_quant_weight_block_grouped(ls.group)


def run_decode(fb, ls, ws):
    for i in range(len(ls.shapes)):
        fb.fp8rl_quant_act_group(ls.X[i], ls.Xq[i], ls.Xs[i])
        fb.fp8rl_gemm_w8a8_block(ls.Xq[i], ls.Xs[i], ls.Wq[i], ls.Ws[i], Y=ls.Y[i], workspace=ws)


def time_step_7b(fb, dev, steps=200):
    """The Qwen2.5-7B layer set at decode M = 64 with a per-step requant: one
    CUDA graph per step (requant of copy s%4, act quant + GEMMs of copy
    (s+2)%4, whose codes were written two steps -- 1.4 GB of traffic -- earlier),
    then the same steps as three graphs with events between them for the
    per-part breakdown."""
    shapes = synth.QWEN25_7B
    M = DECODE_M
    sets = [LayerSet(shapes, M, synth.seed_for(2, 0) + 1000 * c, dev) for c in range(COPIES)]
    ws_bytes = max(fb.fp8rl_gemm_workspace_bytes(M, s.N, s.K) for s in shapes)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    for c in range(COPIES):
        run_requant(fb, sets[c])
        run_decode(fb, sets[c], ws)
    torch.cuda.synchronize()

    def aq(ls):
        for i in range(len(shapes)):
            fb.fp8rl_quant_act_group(ls.X[i], ls.Xq[i], ls.Xs[i])

    def gemm(ls):                      # its codes were written two steps earlier: stable
        for i in range(len(shapes)):
            fb.fp8rl_gemm_w8a8_block(ls.Xq[i], ls.Xs[i], ls.Wq[i], ls.Ws[i], Y=ls.Y[i], workspace=ws,
                                     weights_stable=True)

    g_step = [capture_graph(lambda r=r: (run_requant(fb, sets[r]), aq(sets[(r + COPIES // 2) % COPIES]),
                                         gemm(sets[(r + COPIES // 2) % COPIES])))
              for r in range(COPIES)]
    g_req = [capture_graph(lambda ls=ls: run_requant(fb, ls)) for ls in sets]
    g_aq = [capture_graph(lambda ls=ls: aq(ls)) for ls in sets]
    g_gemm = [capture_graph(lambda ls=ls: gemm(ls)) for ls in sets]
    stream = torch.cuda.current_stream()
    for s in range(5):
        g_step[s % COPIES].replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(steps):
        g_step[s % COPIES].replay()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for s in range(steps):
        r, d = s % COPIES, (s + COPIES // 2) % COPIES
        ev[s][0].record(stream)
        g_req[r].replay()
        ev[s][1].record(stream)
        g_aq[d].replay()
        ev[s][2].record(stream)
        g_gemm[d].replay()
        ev[s][3].record(stream)
    torch.cuda.synchronize()
    req_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    aq_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    gm_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    assert fb.fp8rl_check_device_error() == 0
    sb = step_bytes(shapes, M)
    req_b = sum(requant_bytes(s.N, s.K) for s in shapes)
    gemm_b = sum(gemm_bytes(M, s.N, s.K) for s in shapes)
    aq_b = sum(act_quant_bytes(M, s.K) for s in shapes)
    del g_step, g_req, g_aq, g_gemm, sets
    torch.cuda.empty_cache()
    return {"ms_per_step": ms, "gbs": sb / (ms * 1e-3) / 1e9, "step_bytes": sb,
            "requant_ms": req_ms, "requant_gbs": req_b / (req_ms * 1e-3) / 1e9,
            "act_quant_ms": aq_ms, "act_quant_gbs": aq_b / (aq_ms * 1e-3) / 1e9,
            "gemm_ms": gm_ms, "gemm_gbs": gemm_b / (gm_ms * 1e-3) / 1e9, "steps": steps,
            "workload": "Qwen2.5-7B layer set (qkv 3584->4608, o_proj 3584->3584, gate_up 3584->37888, "
                        "down 18944->3584), decode M=64, per-step requant; one graph per step over 4 rotating "
                        "copies (0.7 GB each)"}


# ------------------------------------------------------------------ extras

def quantization_error(fb, dev):
    """For information: the 8-bit linear layers against the unquantized bf16
    matmul (fp32 accumulation by torch) on the Qwen2.5-7B layer set at M = 64.
    Relative Frobenius error of Y and the largest |error| over rms(Y_ref)."""
    res = {}
    for i, s in enumerate(synth.QWEN25_7B):
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(2, 0) + i, device=dev)
        X = synth.activation(DECODE_M, s.K, synth.seed_for(2, 1) + i, device=dev)
        ref = X.float() @ W.float().t()
        Wq, Ws = fb.fp8rl_quant_weight_block(W)
        y8 = fb.fp8rl_linear_w8a8_block(X, Wq, Ws).float()
        Wi, Wsi = fb.int8rl_quant_weight_channel(W)
        Xi, Xsi = fb.int8rl_quant_act_token(X)
        yi = fb.int8rl_gemm_w8a8(Xi, Xsi, Wi, Wsi).float()
        rms = ref.pow(2).mean().sqrt()
        res[s.name] = {"fp8_rel_fro": float((y8 - ref).norm() / ref.norm()),
                       "fp8_max_over_rms": float((y8 - ref).abs().max() / rms),
                       "int8_rel_fro": float((yi - ref).norm() / ref.norm()),
                       "int8_max_over_rms": float((yi - ref).abs().max() / rms)}
        del W, X, ref, Wq, Ws, Wi, Wsi, Xi, Xsi
    return res


def act_quant_prefill(fb, dev):
    """A2 / A6 at their prefill sizes, where they are HBM-bound: FP8 1x128
    groups at M=8192 and INT8 per token at M=4096, K = 5120 and 27648.  The
    calls walk distinct input copies (> 3x L2) in one graph."""
    hbm = load_peaks()["hbm_gbs"]
    aq = {}
    for K in (5120, 27648):
        for kind, M in (("fp8_group", synth.PREFILL_M), ("int8_token", 4096)):
            nc = _copies_for(2 * M * K)
            Xc = [synth.activation(M, K, synth.seed_for(4, 1), device=dev)]
            Xc += [Xc[0].clone() for _ in range(nc - 1)]
            if kind == "fp8_group":
                Xq = torch.empty(M, K, dtype=torch.uint8, device=dev)
                Xs = torch.empty(K // 128, M, dtype=torch.float32, device=dev)
                ms = _time_graph([lambda c=c: fb.fp8rl_quant_act_group(Xc[c], Xq, Xs) for c in range(nc)])
                nbytes = act_quant_bytes(M, K)
            else:
                Xq = torch.empty(M, K, dtype=torch.int8, device=dev)
                Xs = torch.empty(M, dtype=torch.float32, device=dev)
                ms = _time_graph([lambda c=c: fb.int8rl_quant_act_token(Xc[c], Xq, Xs) for c in range(nc)])
                nbytes = 3 * M * K + 4 * M
            gbs = nbytes / (ms * 1e-3) / 1e9
            aq[f"{kind}_M{M}_K{K}"] = {"us": ms * 1e3, "gbs": gbs, "frac_of_measured_hbm": gbs / hbm,
                                       "input_copies": nc}
            del Xc, Xq, Xs
    return aq


def extras(fb, dev, reps=5):
    out = {}
    out["error_vs_unquantized_bf16_7b_m64"] = quantization_error(fb, dev)
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush = lambda: _flush_l2(flush_buf)  # noqa: E731

    out["act_quant_prefill"] = act_quant_prefill(fb, dev)

    out["qwen7b_decode_step_m64"] = time_step_7b(fb, dev)

    # Grouped MoE GEMM: 64 decode tokens routed top-8 over 128 experts of a
    # hidden-2048 / expert-FFN-768 MoE layer (gate_up N=1536 K=2048, down
    # N=2048 K=768); bytes = the active experts' weights + scales + X + Y
    moe = {}
    E, topk = 128, 8
    rng = torch.Generator().manual_seed(synth.seed_for(8, 0))
    picks = torch.stack([torch.randperm(E, generator=rng)[:topk] for _ in range(DECODE_M)])
    counts = torch.bincount(picks.flatten(), minlength=E)
    offs = torch.cat([torch.zeros(1, dtype=torch.int64), counts.cumsum(0)]).to(torch.int32).to(dev)
    T, active, bound = int(counts.sum()), int((counts > 0).sum()), int(counts.max())
    for name, N, K in (("gate_up", 1536, 2048), ("down", 2048, 768)):
        W = synth.weight_bf16_direct(E * N, K, synth.seed_for(8, 1), device=dev)
        Wq, Ws = fb.fp8rl_quant_weight_block(W)          # stacked experts: per-expert blocks
        del W
        nc = _copies_for(active * N * K)
        Wqs = [Wq.view(E, N, K)] + [Wq.view(E, N, K).clone() for _ in range(nc - 1)]
        Wss = [Ws.view(E, N // 128, K // 128)] + [Ws.view(E, N // 128, K // 128).clone() for _ in range(nc - 1)]
        X = synth.activation(T, K, synth.seed_for(8, 2), device=dev)
        Xq, Xs = fb.fp8rl_quant_act_group(X)
        Y = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
        ms = _time_graph([lambda c=c: fb.fp8rl_gemm_w8a8_block_grouped(Xq, Xs, Wqs[c], Wss[c], offs, bound, Y=Y)
                          for c in range(nc)])
        nbytes = active * (N * K + 4 * (N // 128) * (K // 128)) + T * K + 4 * T * (K // 128) + 2 * T * N
        moe[name] = {"us": ms * 1e3, "gbs": nbytes / (ms * 1e-3) / 1e9, "experts": E, "experts_active": active,
                     "routed_rows": T, "max_rows_per_expert": bound, "weight_copies": nc}
        del Wq, Ws, Wqs, Wss, X, Xq, Xs, Y
    out["moe_fp8_grouped_decode"] = moe

    # Rollout mismatch (FlashRL write-up, Fig. 2, right): KL between the bf16
    # policy's next-token distribution and the FP8 / INT8 rollout's, on a
    # synthetic Qwen2.5-7B LM head (hidden 3584 -> vocab 152064), 64 tokens.  The
    # bf16 reference logits stand for the trainer's forward (torch matmul); the
    # 8-bit logits and the KL come from this library.
    V, K = 152064, 3584
    W = synth.weight_bf16_direct(V, K, synth.seed_for(9, 0), device=dev)
    X = synth.activation(DECODE_M, K, synth.seed_for(9, 1), device=dev)
    R = X @ W.t()
    Wq, Ws = fb.fp8rl_quant_weight_block(W)
    Y8 = fb.fp8rl_linear_w8a8_block(X, Wq, Ws)
    del Wq, Ws
    Wi, Wsi = fb.int8rl_quant_weight_channel(W)
    Xi, Xsi = fb.int8rl_quant_act_token(X)
    Yi = fb.int8rl_gemm_w8a8(Xi, Xsi, Wi, Wsi)
    del W, Wi
    kl8 = fb.fp8rl_logits_kl(R, Y8)
    kli = fb.fp8rl_logits_kl(R, Yi)
    klw = torch.empty(max(1, fb.fp8rl_logits_kl_workspace_bytes(DECODE_M, V)), dtype=torch.uint8, device=dev)
    ms = _time_graph([lambda: fb.fp8rl_logits_kl(R, Y8, kl8, workspace=klw)] * 8)
    out["mismatch_kl_lm_head_7b"] = {
        "tokens": DECODE_M, "vocab": V, "hidden": K,
        "kl_fp8_mean": float(kl8.double().mean()), "kl_int8_mean": float(kli.double().mean()),
        "kl_fp8_max": float(kl8.max()), "kl_int8_max": float(kli.max()),
        "int8_over_fp8": float(kli.double().mean() / kl8.double().mean()),
        "kl_kernel_us": ms * 1e3, "kl_kernel_gbs": 4 * DECODE_M * V / (ms * 1e-3) / 1e9}
    del R, Y8, Yi, X, Xi

    # FP8 KV-cache quant with a per-tensor scale recalibrated each step (32B: 8 kv heads x 128)
    kv = {}
    for tokens in (8192, 32768, 64 * 2048):
        X = synth.activation(tokens, 1024, synth.seed_for(6, 0), device=dev)
        Xq = torch.empty(tokens, 1024, dtype=torch.uint8, device=dev)
        sc = torch.empty(1, dtype=torch.float32, device=dev)
        wsb = torch.empty(max(1, fb.fp8rl_kv_workspace_bytes(tokens, 1024)), dtype=torch.uint8, device=dev)
        nc = _copies_for(2 * tokens * 1024)
        Xc = [X] + [X.clone() for _ in range(nc - 1)]
        ms = _time_graph([lambda c=c: fb.fp8rl_quant_kv_tensor(Xc[c], Xq, sc, workspace=wsb) for c in range(nc)])
        ms2 = _time_graph([lambda c=c: fb.fp8rl_quant_kv_with_scale(Xc[c], sc, Xq) for c in range(nc)])
        b = 3 * tokens * 1024 + 4
        kv[f"tokens{tokens}"] = {"recalibrate_us": ms * 1e3, "recalibrate_gbs": b / (ms * 1e-3) / 1e9,
                                 "with_scale_us": ms2 * 1e3, "with_scale_gbs": b / (ms2 * 1e-3) / 1e9}
        del X, Xc, Xq
    out["kv_cache_fp8_32b"] = kv

    # token-level TIS / MIS weights for a rollout batch (1024 sequences x 16384 tokens)
    n = 1024 * 16384
    g = torch.Generator(device=dev)
    g.manual_seed(synth.seed_for(7, 0))
    lt = torch.randn(n, device=dev, generator=g) - 2.0
    lr = lt + 0.3 * torch.randn(n, device=dev, generator=g)
    mask = torch.ones(n, dtype=torch.uint8, device=dev)
    w = torch.empty(n, dtype=torch.float32, device=dev)
    st = torch.empty(4, dtype=torch.float64, device=dev)
    wsb = torch.empty(max(1, fb.fp8rl_rollout_is_workspace_bytes(n)), dtype=torch.uint8, device=dev)
    out["rollout_is"] = {}
    for mode, name in ((0, "tis"), (1, "mis")):
        ms = _time_graph([lambda: fb.fp8rl_rollout_is_weights(lt, lr, mask, 0.6931472, mode, w, st, wsb)] * 4)
        out["rollout_is"][name] = {"tokens": n, "us": ms * 1e3, "gbs": 13 * n / (ms * 1e-3) / 1e9}
    del lt, lr, mask, w

    # A5-A7: INT8 on the 32B shapes
    i8 = {}
    for s in synth.QWEN25_32B:
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(5, 0), device=dev)
        nc = _copies_for(2 * s.N * s.K)
        Wc = [W] + [W.clone() for _ in range(nc - 1)]
        Wq = torch.empty(s.N, s.K, dtype=torch.int8, device=dev)
        Ws = torch.empty(s.N, dtype=torch.float32, device=dev)
        wq_ms = _time_graph([lambda c=c: fb.int8rl_quant_weight_channel(Wc[c], Wq, Ws) for c in range(nc)])
        i8[f"{s.name}_wquant"] = {"us": wq_ms * 1e3, "gbs": (3 * s.N * s.K + 4 * s.N) / (wq_ms * 1e-3) / 1e9}
        del W, Wc
        nc = _copies_for(s.N * s.K)
        Wqs = [Wq] + [Wq.clone() for _ in range(nc - 1)]
        # the INT8 sweep's sizes, and 128 tokens between them (the 256-token
        # kernel's one-half form)
        for M in sorted(set(synth.INT8_M_SWEEP) | {128}):
            X = synth.activation(M, s.K, synth.seed_for(5, 1), device=dev)
            Xq, Xs = fb.int8rl_quant_act_token(X)
            Y = torch.empty(M, s.N, dtype=torch.bfloat16, device=dev)
            iws = torch.empty(max(16, fb.int8rl_gemm_workspace_bytes(M, s.N, s.K)), dtype=torch.uint8, device=dev)
            if M <= 256:
                ms = _time_graph([lambda c=c: fb.int8rl_gemm_w8a8(Xq, Xs, Wqs[c], Ws, Y=Y, workspace=iws)
                                  for c in range(nc)])
            else:
                ms = _time_op(lambda: fb.int8rl_gemm_w8a8(Xq, Xs, Wq, Ws, Y=Y, workspace=iws), reps, flush)
            del iws
            i8[f"{s.name}_M{M}"] = {"gemm_us": ms * 1e3,
                                    "gemm_gbs": int8_gemm_bytes(M, s.N, s.K) / (ms * 1e-3) / 1e9,
                                    "gemm_tops": 2 * M * s.N * s.K / (ms * 1e-3) / 1e12}
        del Wq, Ws, Wqs
    out["int8_32b"] = i8
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ CPU oracle

class OracleSample:
    """The CPU oracle on a bounded sample of the headline step, with the same
    fraction (about 1/8192) of every part:
      - requant: one 128-row strip per Qwen2.5-32B shape whose block count is
        that shape's share of the 64-layer model's 1 904 640 blocks / 8192
        (18 + 12 + 135 + 68 blocks), seeded bf16 weights after a policy update;
      - act quant: one of the 8192 prefill tokens per shape;
      - GEMM: that token against a full weight per shape.  The GEMM's cost does
        not depend on the values, so its weight operand is seeded random E4M3
        codes and scales (the full 32B weights would take minutes to quantize
        on the host).
    A step runs each part's calls on `threads` host threads (the oracle is
    plain single-threaded C; the calls on disjoint slices run in parallel
    through ctypes, which releases the GIL).  The full-step time is each part's
    measured time divided by its exact fraction."""

    def __init__(self, threads=1):
        import numpy as np

        import oracle
        oracle.build()
        self.np, self.oracle = np, oracle
        self.threads = max(1, threads)
        self.shapes = synth.QWEN25_32B
        total_blocks = LAYERS * sum((s.N // 128) * (s.K // 128) for s in self.shapes)
        self.strips, self.gemm_ops = [], []
        rng = np.random.default_rng(synth.seed_for(4, 9))
        req_blocks = 0
        for i, s in enumerate(self.shapes):
            share = LAYERS * (s.N // 128) * (s.K // 128)
            nb = max(1, round(share / PREFILL_M))
            req_blocks += nb
            W = synth.weight(128, nb * 128, synth.seed_for(4, 0) + 7 * i)
            synth.policy_update_(W, synth.seed_for(4, 0) + 7 * i + 500)
            self.strips.append(synth.bf16_bits(W))
            X = synth.bf16_bits(synth.activation(1, s.K, synth.seed_for(4, 1) + i))
            wq = rng.integers(0, 0x7E, size=(s.N, s.K), dtype=np.uint8)
            wq |= (rng.integers(0, 2, size=(s.N, s.K), dtype=np.uint8) << 7)
            ws = (rng.random((s.N // 128, s.K // 128)) * 1e-3 + 1e-5).astype(np.float32)
            self.gemm_ops.append((X, wq, ws))
        self.f_req = req_blocks / total_blocks
        self.f_tok = 1.0 / PREFILL_M
        self.sample_bytes = (sum(requant_bytes(128, w.shape[1]) for w in self.strips)
                             + sum(act_quant_bytes(1, s.K) for s in self.shapes)
                             + sum(gemm_bytes(PREFILL_M, s.N, s.K) for s in self.shapes) / PREFILL_M)
        self.pool = None
        self.set_threads(self.threads)

    def set_threads(self, threads):
        if self.pool is not None:
            self.pool.shutdown()
        self.threads = max(1, threads)
        self.pool = cf.ThreadPoolExecutor(self.threads) if self.threads > 1 else None

    def _run(self, jobs):
        if self.pool is None:
            return [j() for j in jobs]
        return list(self.pool.map(lambda j: j(), jobs))

    def _split(self, n, unit):
        """Ranges of [0, n) in multiples of `unit`, one per thread (fewer if short)."""
        parts = max(1, min(self.threads, n // unit))
        step = -(-(n // unit) // parts) * unit
        return [(a, min(n, a + step)) for a in range(0, n, step)]

    def step(self):
        np, oracle = self.np, self.oracle
        t = {}
        a = time.perf_counter()
        jobs = []
        for W in self.strips:
            for c0, c1 in self._split(W.shape[1], 128):
                jobs.append(lambda W=W, c0=c0, c1=c1: oracle.fp8_quant_weight_block(np.ascontiguousarray(W[:, c0:c1])))
        self._run(jobs)
        t["requant"] = time.perf_counter() - a
        a = time.perf_counter()
        codes = self._run([lambda X=X: oracle.fp8_quant_act_group(X) for X, _, _ in self.gemm_ops])
        t["act_quant"] = time.perf_counter() - a
        a = time.perf_counter()
        jobs = []
        for (xq, xs), (_, wq, ws) in zip(codes, self.gemm_ops):
            for n0, n1 in self._split(wq.shape[0], 128):
                jobs.append(lambda xq=xq, xs=xs, wq=wq, ws=ws, n0=n0, n1=n1:
                            oracle.fp8_gemm(xq, xs, wq[n0:n1], ws[n0 // 128:n1 // 128]))
        self._run(jobs)
        t["gemm"] = time.perf_counter() - a
        return t

    def full_step_seconds(self, t):
        return {"requant": t["requant"] / self.f_req, "act_quant": t["act_quant"] / self.f_tok,
                "gemm": t["gemm"] / self.f_tok}

    def describe(self):
        return (f"per sample step: the oracle's requant of 233 of the 64-layer Qwen2.5-32B model's 1904640 "
                f"weight blocks (128-row strips, each shape's share), act quant of 1 of the 8192 prefill "
                f"tokens per shape and that token's GEMM against full 32B weights (seeded random codes); "
                f"{self.threads} host thread(s); value = full-step bytes / full-step time extrapolated by "
                f"each part's fraction (requant {self.f_req:.3g}, tokens {self.f_tok:.3g})")

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()


def _oracle_rate(o, threads, n_steps):
    o.set_threads(threads)
    o.step()                                            # warm-up (page-in, thread start)
    tot = {"requant": 0.0, "act_quant": 0.0, "gemm": 0.0}
    sample_s = []
    for _ in range(n_steps):
        t = o.step()
        sample_s.append(sum(t.values()))
        for k, v in o.full_step_seconds(t).items():
            tot[k] += v / n_steps
    full = sum(tot.values())
    return {"value": model_step_bytes() / full / 1e9, "full_step_seconds": tot,
            "sample_step_seconds": statistics.mean(sample_s), "sample_steps": n_steps,
            "sample": o.describe()}


def cpu_baseline(n_single=8, n_all=20):
    """The oracle on the machine's host cores: one thread, and every core of the
    process's affinity mask (about 10-20 s in all)."""
    cores = host_cores()
    o = OracleSample(1)
    one = _oracle_rate(o, 1, n_single)
    alln = _oracle_rate(o, cores, n_all)
    o.close()
    return {"value": alln["value"], "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": alln["sample"], "extrapolated": True, "cpu_model": cpu_model(),
            "sample_step_seconds": alln["sample_step_seconds"], "full_step_seconds": alln["full_step_seconds"],
            "single_thread": {"value": one["value"], "cores": 1,
                              "sample_step_seconds": one["sample_step_seconds"],
                              "full_step_seconds": one["full_step_seconds"]}}


def main_reference(args, world, rank):
    """The oracle as the reference arm: every step is one bounded sample of the
    headline step on all of the host's cores; ms_per_step is the sample's own
    measured time and value the full-step rate extrapolated from it."""
    if rank != 0:
        return 0
    cores = host_cores()
    o = OracleSample(cores)
    for _ in range(args.warmup):
        o.step()
    t0 = time.perf_counter()
    samples = [o.step() for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    o.close()
    full = statistics.mean(sum(o.full_step_seconds(t).values()) for t in samples)
    sample_ms = statistics.mean(sum(t.values()) for t in samples) * 1e3
    v = model_step_bytes() / full / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sample_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic", "config": workload_config(),
            "extrapolated": True, "full_step_seconds_extrapolated": full,
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": o.describe(),
                             "extrapolated": True, "cpu_model": cpu_model(), "sample_step_ms": sample_ms},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)
    return 0


def workload_config():
    return {"workload": "Qwen2.5-32B-shaped model: per-step FP8 128x128 requant of all 64 layers "
                        "(qkv 5120->7168, o_proj 5120->5120, gate_up 5120->55296, down 27648->5120; 256 "
                        "tensors, 62.4 GB bf16) after W += N(0,1e-4), then act quant + FP8 block-scaled "
                        "GEMM at prefill M=8192 for each layer shape",
            "M": PREFILL_M, "layers": LAYERS, "shapes": [[s.name, s.K, s.N] for s in synth.QWEN25_32B],
            "l2": "inputs larger than L2: 62.4 GB of weights and 31.2 GB of codes per step",
            "parallelism": "replicas"}



def profile_case(fb, case, dev, reps=3):
    """Small, self-contained workloads for ncu captures (a few GB at most, a
    few launches of one kernel)."""
    if case == "requant":
        ls = LayerSet(synth.QWEN25_7B, DECODE_M, synth.seed_for(2, 0), dev)
        for _ in range(reps):
            run_requant(fb, ls)
    elif case in ("decode", "act_quant"):
        ls = LayerSet(synth.QWEN25_7B, DECODE_M, synth.seed_for(2, 0), dev)
        run_requant(fb, ls)
        ws = torch.empty(max(1, max(fb.fp8rl_gemm_workspace_bytes(DECODE_M, s.N, s.K) for s in ls.shapes)),
                         dtype=torch.uint8, device=dev)
        for _ in range(reps):
            run_decode(fb, ls, ws)
    elif case.startswith("decode7b_m"):
        M = int(case[len("decode7b_m"):])
        s = synth.QWEN25_7B[2]                          # gate_up 3584 -> 37888
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(2, 0), device=dev)
        Wq, Ws = fb.fp8rl_quant_weight_block(W)
        del W
        Xq, Xs = fb.fp8rl_quant_act_group(synth.activation(M, s.K, synth.seed_for(2, 1), device=dev))
        for _ in range(reps):
            fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws)
    elif case.startswith("decode7b_qkv_m"):
        M = int(case[len("decode7b_qkv_m"):])
        s = synth.QWEN25_7B[0]                          # qkv 3584 -> 4608
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(2, 0), device=dev)
        Wq, Ws = fb.fp8rl_quant_weight_block(W)
        del W
        Xq, Xs = fb.fp8rl_quant_act_group(synth.activation(M, s.K, synth.seed_for(2, 1), device=dev))
        ws = torch.empty(max(16, fb.fp8rl_gemm_workspace_bytes(M, s.N, s.K)), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws, workspace=ws)
    elif case.startswith("int8_qkv_m"):
        M = int(case[len("int8_qkv_m"):])
        s = synth.QWEN25_32B[0]                         # qkv 5120 -> 7168
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(5, 0), device=dev)
        Wq, Ws = fb.int8rl_quant_weight_channel(W)
        del W
        Xq, Xs = fb.int8rl_quant_act_token(synth.activation(M, s.K, synth.seed_for(5, 1), device=dev))
        ws = torch.empty(max(16, fb.int8rl_gemm_workspace_bytes(M, s.N, s.K)), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            fb.int8rl_gemm_w8a8(Xq, Xs, Wq, Ws, workspace=ws)
    elif case.startswith("decode7b_down_m"):
        M = int(case[len("decode7b_down_m"):])
        s = synth.QWEN25_7B[3]                          # down 18944 -> 3584
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(2, 0), device=dev)
        Wq, Ws = fb.fp8rl_quant_weight_block(W)
        del W
        Xq, Xs = fb.fp8rl_quant_act_group(synth.activation(M, s.K, synth.seed_for(2, 1), device=dev))
        ws = torch.empty(max(16, fb.fp8rl_gemm_workspace_bytes(M, s.N, s.K)), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws, workspace=ws)
    elif case.startswith("prefill_down_m"):
        M = int(case[len("prefill_down_m"):])
        s = synth.QWEN25_32B[3]                         # down 27648 -> 5120
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(4, 0), device=dev)
        Wq, Ws = fb.fp8rl_quant_weight_block(W)
        del W
        Xq, Xs = fb.fp8rl_quant_act_group(synth.activation(M, s.K, synth.seed_for(4, 1), device=dev))
        ws = torch.empty(max(16, fb.fp8rl_gemm_workspace_bytes(M, s.N, s.K)), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws, workspace=ws)
    elif case.startswith("decode32b_m"):
        M = int(case[len("decode32b_m"):])
        s = synth.QWEN25_32B[2]                         # gate_up 5120 -> 55296
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(3, 0), device=dev)
        Wq, Ws = fb.fp8rl_quant_weight_block(W)
        del W
        Xq, Xs = fb.fp8rl_quant_act_group(synth.activation(M, s.K, synth.seed_for(3, 1), device=dev))
        for _ in range(reps):
            fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws)
    elif case in ("moe", "moe_down"):
        E = 128                                          # top-8 of 64 tokens
        N, K = (1536, 2048) if case == "moe" else (2048, 768)   # gate_up / down
        rng = torch.Generator().manual_seed(synth.seed_for(8, 0))
        picks = torch.stack([torch.randperm(E, generator=rng)[:8] for _ in range(DECODE_M)])
        counts = torch.bincount(picks.flatten(), minlength=E)
        offs = torch.cat([torch.zeros(1, dtype=torch.int64), counts.cumsum(0)]).to(torch.int32).to(dev)
        W = synth.weight_bf16_direct(E * N, K, synth.seed_for(8, 1), device=dev)
        Wq, Ws = fb.fp8rl_quant_weight_block(W)
        del W
        Xq, Xs = fb.fp8rl_quant_act_group(synth.activation(int(counts.sum()), K, synth.seed_for(8, 2), device=dev))
        for _ in range(reps):
            fb.fp8rl_gemm_w8a8_block_grouped(Xq, Xs, Wq.view(E, N, K), Ws.view(E, N // 128, K // 128), offs,
                                             int(counts.max()))
    elif case == "kl":
        V = 152064
        g = torch.Generator(device=dev)
        g.manual_seed(synth.seed_for(9, 2))
        R = (2.0 * torch.randn(DECODE_M, V, device=dev, generator=g)).to(torch.bfloat16)
        Q = (R.float() + 0.02 * torch.randn(DECODE_M, V, device=dev, generator=g)).to(torch.bfloat16)
        for _ in range(reps):
            fb.fp8rl_logits_kl(R, Q)
    elif case == "int8_gate_up_m256":                 # A7 on the 256-token kernel
        s = synth.QWEN25_32B[2]                          # gate_up 5120 -> 55296
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(5, 0), device=dev)
        Wq, Ws = fb.int8rl_quant_weight_channel(W)
        del W
        Xq, Xs = fb.int8rl_quant_act_token(synth.activation(256, s.K, synth.seed_for(5, 1), device=dev))
        ws = torch.empty(max(16, fb.int8rl_gemm_workspace_bytes(256, s.N, s.K)), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            fb.int8rl_gemm_w8a8(Xq, Xs, Wq, Ws, workspace=ws)
    elif case == "int8_m32":
        s = synth.QWEN25_32B[2]                          # gate_up 5120 -> 55296
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(5, 0), device=dev)
        Wq, Ws = fb.int8rl_quant_weight_channel(W)
        del W
        Xq, Xs = fb.int8rl_quant_act_token(synth.activation(32, s.K, synth.seed_for(5, 1), device=dev))
        for _ in range(reps):
            fb.int8rl_gemm_w8a8(Xq, Xs, Wq, Ws)
    elif case == "kv":
        X = synth.activation(64 * 2048, 1024, synth.seed_for(6, 0), device=dev)
        for _ in range(reps):
            fb.fp8rl_quant_kv_tensor(X)
    elif case == "act_quant_prefill":                 # A2 at M=8192, K=27648: four groups per thread
        X = synth.activation(synth.PREFILL_M, 27648, synth.seed_for(4, 1), device=dev)
        Xq = torch.empty(synth.PREFILL_M, 27648, dtype=torch.uint8, device=dev)
        Xs = torch.empty(27648 // 128, synth.PREFILL_M, dtype=torch.float32, device=dev)
        for _ in range(reps):
            fb.fp8rl_quant_act_group(X, Xq, Xs)
    elif case == "kv8192":                            # one cooperative pass (fits the resident CTAs)
        X = synth.activation(8192, 1024, synth.seed_for(6, 0), device=dev)
        ws = torch.empty(fb.fp8rl_kv_workspace_bytes(8192, 1024), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            fb.fp8rl_quant_kv_tensor(X, workspace=ws)
    elif case == "tis":
        n = 1024 * 16384
        lt = torch.randn(n, device=dev) - 2.0
        lr = lt + 0.3 * torch.randn(n, device=dev)
        for _ in range(reps):
            fb.fp8rl_rollout_is_weights(lt, lr, None, 0.6931472, 0)
    elif case == "prefill":
        s = synth.QWEN25_32B[0]
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(4, 0), device=dev)
        Wq, Ws = fb.fp8rl_quant_weight_block(W)
        Xq, Xs = fb.fp8rl_quant_act_group(synth.activation(synth.PREFILL_M, s.K, synth.seed_for(4, 1), device=dev))
        ws = torch.empty(max(1, fb.fp8rl_gemm_workspace_bytes(synth.PREFILL_M, s.N, s.K)), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws, workspace=ws)
    elif case == "int8":
        s = synth.QWEN25_32B[0]
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(5, 0), device=dev)
        Wq, Ws = fb.int8rl_quant_weight_channel(W)
        Xq, Xs = fb.int8rl_quant_act_token(synth.activation(256, s.K, synth.seed_for(5, 1), device=dev))
        for _ in range(reps):
            fb.int8rl_gemm_w8a8(Xq, Xs, Wq, Ws)
    elif case.startswith("requant32b_layers"):         # A1 over a few 32B layers in one grouped launch
        n = int(case[len("requant32b_layers"):])
        items = []
        for layer in range(n):
            for i, s in enumerate(synth.QWEN25_32B):
                W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(4, 0) + 1000 * layer + i, device=dev)
                items.append((W, torch.empty(s.N, s.K, dtype=torch.uint8, device=dev),
                              torch.empty(s.N // 128, s.K // 128, dtype=torch.float32, device=dev)))
        req = fb.GroupedRequant(items)
        for _ in range(reps):
            req()
    elif case == "prefill32b":                         # A3: one launch per 32B shape at M=8192
        for s in synth.QWEN25_32B:
            W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(4, 0), device=dev)
            Wq, Ws = fb.fp8rl_quant_weight_block(W)
            del W
            Xq, Xs = fb.fp8rl_quant_act_group(synth.activation(synth.PREFILL_M, s.K, synth.seed_for(4, 1),
                                                                device=dev))
            ws = torch.empty(max(16, fb.fp8rl_gemm_workspace_bytes(synth.PREFILL_M, s.N, s.K)),
                             dtype=torch.uint8, device=dev)
            fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws, workspace=ws)
            torch.cuda.synchronize()
            del Wq, Ws, Xq, Xs, ws
    elif case.startswith("decode32b_") and "_m" in case:   # A4: decode32b_<shape>_m<M>
        name, m = case[len("decode32b_"):].rsplit("_m", 1)
        s = {x.name: x for x in synth.QWEN25_32B}[name]
        M = int(m)
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(3, 0), device=dev)
        Wq, Ws = fb.fp8rl_quant_weight_block(W)
        del W
        Xq, Xs = fb.fp8rl_quant_act_group(synth.activation(M, s.K, synth.seed_for(3, 1), device=dev))
        ws = torch.empty(max(16, fb.fp8rl_gemm_workspace_bytes(M, s.N, s.K)), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws, workspace=ws)
    else:
        raise SystemExit(f"unknown profile case {case}")
    torch.cuda.synchronize()
    assert fb.fp8rl_check_device_error() == 0
    print(f"profile case {case}: ok")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--extras", default="all", choices=["all", "none"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--clocks-out", default=None,
                    help="CSV path for the nvidia-smi clock samples of the timed region (default: a temp file)")
    ap.add_argument("--profile", default=None,
                    help="run one small case for ncu: requant | requant32b_layers<n> | prefill32b | "
                         "decode32b_<shape>_m<M> | decode | decode7b_m<M> | decode7b_qkv_m<M> | "
                         "decode7b_down_m<M> | decode32b_m<M> | prefill | prefill_down_m<M> | int8 | int8_m32 | "
                         "int8_qkv_m<M> | int8_gate_up_m256 | kv | kv8192 | tis | moe | moe_down | kl | act_quant_prefill")
    args = ap.parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        return main_reference(args, world, rank)
    if args.warmup < 3:
        print("note: warm-up raised to the minimum of 3 steps", file=sys.stderr)
        args.warmup = 3

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    from precision_rl_rollout_gb300 import binding as fb
    fb.load()
    if args.profile:
        return profile_case(fb, args.profile, dev)

    model = Model32B(fb, dev)
    torch.cuda.synchronize()
    head = time_headline(fb, args, dev, world, rank, model)
    e2e = None if args.no_e2e else time_e2e(fb, args, dev, model)
    del model
    torch.cuda.empty_cache()
    dec = decode_sweep_32b(fb, dev)

    parts = model_step_parts()
    sb = model_step_bytes()
    ms_per_step = head["total_ms"] / args.steps
    value = world * sb / (ms_per_step * 1e-3) / 1e9
    peaks = load_peaks()
    roof = roofline_entries(head, dec, peaks)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": workload_config(),
            "roofline": roof,
            "breakdown": {"requant_ms": head["req_ms"], "act_quant_ms": head["aq_ms"],
                          "act_quant_gbs": parts["act_quant_bytes"] / (head["aq_ms"] * 1e-3) / 1e9,
                          "gemm_ms": dict(zip([s.name for s in synth.QWEN25_32B], head["gemm_ms"])),
                          "step_ms_p10_p50_p90": head["step_ms_pct"],
                          "step_bytes": sb, "step_parts": parts,
                          "method": "CUDA events between the parts of every timed step, on the launching stream"},
            "decode_sweep_32b": dec,
            "gpu_launches": head["launches_per_step"] * args.steps,
            "clocks": head["clocks"]}
    if e2e is not None:
        line["e2e"] = e2e
    if args.extras == "all" and rank == 0:
        line["extras"] = extras(fb, dev)
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline()
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
