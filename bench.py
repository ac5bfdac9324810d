"""Benchmark of the 8-bit rollout linear-layer hot path on GB300.

Headline (one JSON line on rank 0): the Qwen2.5-7B-shaped layer set (qkv
3584->4608, o_proj 3584->3584, gate_up 3584->37888, down 18944->3584) at decode
batch M=64 with a per-step FP8 weight requant.  One step is one pass of the
FP8 path over that layer set:
  A1  requant all four bf16 weights to 128x128-block E4M3 + fp32 scales
      (one grouped launch),
  A2  quantize the four layer inputs X [64, K] to 1x128-group E4M3,
  A4  run the four block-scaled FP8 GEMMs -> bf16 Y [64, N].
value = algorithmic HBM bytes of the step / step time (GB/s).  Four copies of
the layer set rotate: step s requants copy s%4 and runs the GEMMs on copy
(s+2)%4, whose E4M3 weights were written two steps (1.4 GB of traffic)
earlier, so every weight byte comes from HBM, not from L2.

Other rows are measured as sub-benchmarks under "extras" (not in `value`):
prefill FP8 GEMM TFLOP/s at M=8192 (Qwen2.5-32B shapes), the 32B decode sweep
M in {1,8,32,128,256}, the grouped MoE GEMM, the FP8-vs-INT8 rollout mismatch
KL, the 64-layer 32B requant, the FP8 KV-cache quant, the TIS/MIS weights and
the INT8 W8A8 path.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--extras all|none]
    python bench.py --impl reference ...     # the CPU oracle on a bounded sample
Under torchrun each rank is an independent replica (the path does not shard).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
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

# ncu-measured DRAM traffic of the dominant kernel, valid only for the source it
# was taken on (checked by hash; null otherwise).  Filled from the committed
# profile summary of the same workload.
NCU_TRAFFIC = {"kernel": "quant_weight_block_kernel", "source_sha1": "69912cc3432327fae840b52154efe497e2f08df4",
               "bytes_per_launch": 466135296 + 174760960,
               "profile": "profiles/requant_weight_block_qwen7b.md"}


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
    return sum(requant_bytes(s.N, s.K) + act_quant_bytes(M, s.K) + gemm_bytes(M, s.N, s.K)
               for s in shapes)


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
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int, rank: int = 0):
        self.smi_id = _smi_id(device)
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_rank{rank}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
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
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
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
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ device step

class LayerSet:
    """One copy of the FP8 layer set: bf16 weights, their E4M3 codes and scales,
    the four layer inputs and their quantized forms, and the outputs."""

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


def capture_graph(fn):
    """Capture fn's launches (library calls on the current stream) into a CUDA graph."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def time_headline(fb, args, dev, world, rank):
    shapes = synth.QWEN25_7B
    M = DECODE_M
    sets = [LayerSet(shapes, M, synth.seed_for(2, 0) + 1000 * c, dev) for c in range(COPIES)]
    ws_bytes = max(fb.fp8rl_gemm_workspace_bytes(M, s.N, s.K) for s in shapes)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    # kernels per GEMM call with this workspace (a split added by a second launch counts two)
    gemm_launches = sum(fb.fp8rl_gemm_kernel_count(M, s.N, s.K, ws_bytes) for s in shapes)
    for c in range(COPIES):                          # every copy has valid codes before step 0
        run_requant(fb, sets[c])
        run_decode(fb, sets[c], ws)                  # first calls outside capture (one-time set-up)
    torch.cuda.synchronize()

    def aq(ls):
        for i in range(len(shapes)):
            fb.fp8rl_quant_act_group(ls.X[i], ls.Xq[i], ls.Xs[i])

    def gemm(ls):
        for i in range(len(shapes)):
            fb.fp8rl_gemm_w8a8_block(ls.Xq[i], ls.Xs[i], ls.Wq[i], ls.Ws[i], Y=ls.Y[i], workspace=ws)

    # One graph per step pattern (requant of copy r, then act quant and GEMMs of
    # copy d): the launch cost of the host binding stays out of the step and the
    # kernels chain through programmatic dependent launch across the parts.
    # Separate graphs per part, with events between them, give the breakdown.
    g_step = [capture_graph(lambda r=r: (run_requant(fb, sets[r]), aq(sets[(r + COPIES // 2) % COPIES]),
                                         gemm(sets[(r + COPIES // 2) % COPIES])))
              for r in range(COPIES)]
    g_req = [capture_graph(lambda ls=ls: run_requant(fb, ls)) for ls in sets]
    g_aq = [capture_graph(lambda ls=ls: aq(ls)) for ls in sets]
    g_gemm = [capture_graph(lambda ls=ls: gemm(ls)) for ls in sets]
    stream = torch.cuda.current_stream()

    def step(s):
        g_step[s % COPIES].replay()

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device(), rank) as clk:
        t0.record(stream)
        for s in range(args.steps):
            step(args.warmup + s)
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)

    nb = max(3, min(args.steps, 200))                 # breakdown pass (not the timed region)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nb)]
    for s in range(nb):
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
    res = {"total_ms": total_ms, "req_ms": req_ms, "aq_ms": aq_ms, "gemm_ms": gm_ms,
           "clocks": clk.summary(), "launches_per_step": 1 + len(shapes) + gemm_launches}
    del g_step, g_req, g_aq, g_gemm, sets
    torch.cuda.empty_cache()
    return res


def time_e2e(fb, args, dev):
    """Same step through the public API with pinned host buffers: H2D of the
    bf16 weights and inputs, requant, act quant, GEMM on the fresh codes, D2H
    of Y.  As a user would run it: the copies in, the compute and the copies
    out go on three streams, and two device-side layer sets alternate, so the
    next step's inputs stream in while this step computes (events order every
    reuse of a set's buffers)."""
    shapes = synth.QWEN25_7B
    M = DECODE_M
    sets = [LayerSet(shapes, M, synth.seed_for(2, 0) + 7000 + 100 * c, dev) for c in range(2)]
    hW = [w.cpu().pin_memory() for w in sets[0].W]
    hX = [x.cpu().pin_memory() for x in sets[0].X]
    hY = [[torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in sets[0].Y] for _ in range(2)]
    ws_bytes = max(fb.fp8rl_gemm_workspace_bytes(M, s.N, s.K) for s in shapes)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in hW + hX)
    d2h = sum(t.numel() * t.element_size() for t in hY[0])
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]     # set c's inputs have landed
    ev_done = [torch.cuda.Event() for _ in range(2)]   # set c's compute is done (W, X free; Y ready)
    ev_out = [torch.cuda.Event() for _ in range(2)]    # set c's Y has been read back (Y free)
    for c in range(2):                                 # every event recorded once before first use
        ev_done[c].record(comp)
        ev_out[c].record(comp)

    def step(n):
        c = n % 2
        ls = sets[c]
        s_in.wait_event(ev_done[c])
        with torch.cuda.stream(s_in):
            for i in range(len(shapes)):
                ls.W[i].copy_(hW[i], non_blocking=True)
                ls.X[i].copy_(hX[i], non_blocking=True)
        ev_in[c].record(s_in)
        comp.wait_event(ev_in[c])
        comp.wait_event(ev_out[c])
        run_requant(fb, ls)
        run_decode(fb, ls, ws)
        ev_done[c].record(comp)
        s_out.wait_event(ev_done[c])
        with torch.cuda.stream(s_out):
            for i in range(len(shapes)):
                hY[c][i].copy_(ls.Y[i], non_blocking=True)
        ev_out[c].record(s_out)

    steps = max(3, min(args.steps, 20))
    for n in range(max(3, args.warmup)):
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
    del sets
    torch.cuda.empty_cache()
    return {"value": step_bytes(shapes, M) / (ms * 1e-3) / 1e9, "unit": UNIT,
            "ms_per_step": ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "method": "copies in / compute / copies out on three streams, two device sets alternating"}


# ------------------------------------------------------------------ extras

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

    # A3: prefill FP8 GEMM at M=8192 on the 32B shapes (ms-scale launches)
    pre = {}
    for s in synth.QWEN25_32B:
        W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(4, 0), device=dev)
        Wq, Ws = fb.fp8rl_quant_weight_block(W)
        del W
        X = synth.activation(synth.PREFILL_M, s.K, synth.seed_for(4, 1), device=dev)
        Xq, Xs = fb.fp8rl_quant_act_group(X)
        del X
        Y = torch.empty(synth.PREFILL_M, s.N, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(1, fb.fp8rl_gemm_workspace_bytes(synth.PREFILL_M, s.N, s.K)),
                         dtype=torch.uint8, device=dev)
        ms = _time_op(lambda: fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws, Y=Y, workspace=ws), reps, flush)
        pre[s.name] = {"ms": ms, "tflops": 2 * synth.PREFILL_M * s.N * s.K / (ms * 1e-3) / 1e12}
        del Wq, Ws, Xq, Xs, Y
    out["prefill_fp8_gemm_m8192"] = pre

    out["act_quant_prefill"] = act_quant_prefill(fb, dev)

    # A2 + A4: 32B decode sweep; each GEMM walks distinct weight copies (> 3x L2)
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
            ms = _time_graph([lambda c=c: fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wqs[c], Wss[c], Y=Y, workspace=gws)
                              for c in range(nc)])
            aq = _time_graph([lambda: fb.fp8rl_quant_act_group(X, Xq, Xs)] * 16)
            dec[f"{s.name}_M{M}"] = {"gemm_us": ms * 1e3, "gemm_gbs": gemm_bytes(M, s.N, s.K) / (ms * 1e-3) / 1e9,
                                     "gemm_tflops": 2 * M * s.N * s.K / (ms * 1e-3) / 1e12,
                                     "act_quant_us": aq * 1e3, "weight_copies": nc}
        del Wq, Ws, Wqs, Wss
    out["decode_fp8_gemm_32b"] = dec

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

    # A1 at full-model scale: 64 layers x 4 shapes, grouped launches (62 GB in)
    items = []
    for layer in range(synth.QWEN25_32B_LAYERS):
        for i, s in enumerate(synth.QWEN25_32B):
            W = synth.weight_bf16_direct(s.N, s.K, synth.seed_for(4, 0) + 1000 * layer + i, device=dev)
            items.append((W, torch.empty(s.N, s.K, dtype=torch.uint8, device=dev),
                          torch.empty(s.N // 128, s.K // 128, dtype=torch.float32, device=dev)))
    nbytes = sum(requant_bytes(s.N, s.K) for s in synth.QWEN25_32B) * synth.QWEN25_32B_LAYERS
    ms = _time_op(lambda: fb.fp8rl_quant_weight_block_grouped(items), max(3, reps // 2))
    out["requant_fp8_32b_64layers"] = {"ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9,
                                       "bytes": nbytes, "tensors": len(items)}
    del items
    torch.cuda.empty_cache()

    # FP8 KV-cache quant with a per-tensor scale recalibrated each step (32B: 8 kv heads x 128)
    kv = {}
    for tokens in (8192, 64 * 2048):
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
        for M in synth.INT8_M_SWEEP:
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
    """The CPU oracle on a bounded sample of the headline step.  Set-up (untimed)
    draws the same seeded inputs as the GPU and quantizes the full weights once
    (the GEMM sample needs every weight row).  Each sample step times the
    oracle's requant of `req_rows` rows of every weight, its act quant of all
    four X [64, K] and its GEMM for `gemm_rows` tokens against the full weights,
    then extrapolates each part linearly to the full step."""

    def __init__(self, req_rows=128, gemm_rows=1):
        import numpy as np

        import oracle
        oracle.build()
        self.np, self.oracle = np, oracle
        self.req_rows, self.gemm_rows = req_rows, gemm_rows
        self.shapes = synth.QWEN25_7B
        self.data = []
        for i, s in enumerate(self.shapes):
            W = synth.bf16_bits(synth.weight(s.N, s.K, synth.seed_for(2, 0) + 10 * i))
            X = synth.bf16_bits(synth.activation(DECODE_M, s.K, synth.seed_for(2, 0) + 10 * i + 1))
            wq, ws = oracle.fp8_quant_weight_block(W)
            xq, xs = oracle.fp8_quant_act_group(X)
            self.data.append((W, X, wq, ws, xq, xs))
        self.step_idx = 0

    def step(self):
        np, oracle = self.np, self.oracle
        t = {"requant": 0.0, "act_quant": 0.0, "gemm": 0.0}
        for s, (W, X, wq, ws, xq, xs) in zip(self.shapes, self.data):
            r0 = (self.step_idx * self.req_rows) % s.N
            a = time.perf_counter()
            oracle.fp8_quant_weight_block(np.ascontiguousarray(W[r0:r0 + self.req_rows]))
            t["requant"] += (time.perf_counter() - a) * (s.N / self.req_rows)
            a = time.perf_counter()
            oracle.fp8_quant_act_group(X)
            t["act_quant"] += time.perf_counter() - a
            m0 = (self.step_idx * self.gemm_rows) % DECODE_M
            a = time.perf_counter()
            oracle.fp8_gemm(np.ascontiguousarray(xq[m0:m0 + self.gemm_rows]),
                            np.ascontiguousarray(xs[:, m0:m0 + self.gemm_rows]), wq, ws)
            t["gemm"] += (time.perf_counter() - a) * (DECODE_M / self.gemm_rows)
        self.step_idx += 1
        return t

    def describe(self):
        return (f"per sample step: oracle requant of {self.req_rows} rows of each Qwen2.5-7B weight (scaled "
                f"to all rows), act quant of all four X [64,K], GEMM for {self.gemm_rows} of 64 tokens against "
                f"the full weights (scaled x{DECODE_M // self.gemm_rows}); single-threaded C oracle; value = "
                f"full-step algorithmic bytes / extrapolated full-step time")


def cpu_baseline(n_steps=3, req_rows=1024, gemm_rows=16):
    """About 10-20 s of oracle work on the machine's host cores (1 thread)."""
    o = OracleSample(req_rows=req_rows, gemm_rows=gemm_rows)
    tot = {"requant": 0.0, "act_quant": 0.0, "gemm": 0.0}
    for _ in range(n_steps):
        for k, v in o.step().items():
            tot[k] += v / n_steps
    full = sum(tot.values())
    return {"value": step_bytes(o.shapes, DECODE_M) / full / 1e9, "unit": UNIT, "cores": 1,
            "kind": "oracle", "sample": o.describe() + f"; mean of {n_steps} sample steps",
            "full_step_seconds": tot}


# ------------------------------------------------------------------ main

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


def traffic_or_null():
    sha = requant_source_sha1()
    if NCU_TRAFFIC["source_sha1"] == sha and NCU_TRAFFIC["bytes_per_launch"]:
        return NCU_TRAFFIC["bytes_per_launch"]
    return None


def main_reference(args, world, rank):
    if rank != 0:
        return 0
    o = OracleSample(req_rows=128, gemm_rows=1)
    for _ in range(args.warmup):
        o.step()
    t0 = time.perf_counter()
    full_s = [sum(o.step().values()) for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    shapes = synth.QWEN25_7B
    v = step_bytes(shapes, DECODE_M) / statistics.mean(full_s) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_bytes(shapes, DECODE_M) / (v * 1e9) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic", "config": workload_config(),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": o.describe()},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)
    return 0


def workload_config():
    return {"workload": "Qwen2.5-7B-shaped layer set (qkv 3584->4608, o_proj 3584->3584, gate_up "
                        "3584->37888, down 18944->3584), decode M=64, per-step FP8 128x128 requant",
            "M": DECODE_M, "layers": [[s.name, s.K, s.N] for s in synth.QWEN25_7B],
            "copies": COPIES,
            "l2": "inputs larger than L2: 4 rotating copies (0.7 GB each); GEMM weights written 2 steps earlier",
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
    elif case == "moe":
        E, N, K = 128, 1536, 2048                         # MoE gate_up, top-8 of 64 tokens
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
    else:
        raise SystemExit(f"unknown profile case {case}")
    torch.cuda.synchronize()
    assert fb.fp8rl_check_device_error() == 0
    print(f"profile case {case}: ok")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--extras", default="all", choices=["all", "none"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--profile", default=None,
                    help="run one small case for ncu: requant | decode | decode7b_m<M> | decode7b_qkv_m<M> | "
                         "decode7b_down_m<M> | decode32b_m<M> | prefill | prefill_down_m<M> | int8 | int8_m32 | "
                         "int8_qkv_m<M> | kv | tis | moe | kl")
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

    head = time_headline(fb, args, dev, world, rank)
    shapes = synth.QWEN25_7B
    sb = step_bytes(shapes, DECODE_M)
    ms_per_step = head["total_ms"] / args.steps
    value = world * sb / (ms_per_step * 1e-3) / 1e9
    peaks = load_peaks()
    req_b = sum(requant_bytes(s.N, s.K) for s in shapes)
    req_gbs = req_b / (head["req_ms"] * 1e-3) / 1e9
    gemm_b = sum(gemm_bytes(DECODE_M, s.N, s.K) for s in shapes)
    aq_b = sum(act_quant_bytes(DECODE_M, s.K) for s in shapes)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": workload_config(),
            "roofline": {"bound": "hbm", "kernel": "quant_weight_block_kernel (A1 requant, grouped)",
                         "achieved": req_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": req_gbs / peaks["hbm_gbs"], "traffic": traffic_or_null(),
                         "algorithmic_bytes_per_launch": req_b,
                         "peak_source": f"{peaks['source']} hbm_gbs (STREAM-style copy)"},
            "breakdown": {"requant_ms": head["req_ms"], "requant_gbs": req_gbs,
                          "act_quant_ms": head["aq_ms"], "act_quant_gbs": aq_b / (head["aq_ms"] * 1e-3) / 1e9,
                          "gemm_ms": head["gemm_ms"], "gemm_gbs": gemm_b / (head["gemm_ms"] * 1e-3) / 1e9,
                          "step_bytes": sb,
                          "method": "the timed steps replayed as three graphs (requant | act quant | GEMMs) "
                                    "with CUDA events between them, right after the timed region"},
            "gpu_launches": head["launches_per_step"] * args.steps,
            "clocks": head["clocks"]}
    if not args.no_e2e:
        line["e2e"] = time_e2e(fb, args, dev)
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
