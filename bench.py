#!/usr/bin/env python
"""Benchmark of the fused attention forward on GB300.

Default (one GPU): the GQA causal long prefill B2 Hq32 Hkv8 L8192 d128 bf16
(the largest single-GPU workload; 4 query heads per kv head), metric =
attention-forward TFLOP/s on unmasked (query, key) pairs.  The same run also
measures the other full-size workloads (dense causal prefill B4 H16 L2048,
paged decode in GB/s, varlen soft-cap + sink prefill, the masks, chunked
prefill, FP8) and reports them under "extra".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: W untimed warm-up steps, then K timed steps.  A step is `passes`
back-to-back passes of the whole hot path over the workload (each pass one
call of the public entry point on inputs resident in HBM), enough passes that
the timed loop lasts about --min-seconds of wall time so the clocks are
sampled under load.  Before every pass a 256 MiB buffer is written so L2
(129 MB) holds nothing of the inputs; each pass is bracketed by CUDA events
recorded on the launching stream (the flush lies outside them); the timed
loop is bracketed by a barrier and a device synchronise.  nvidia-smi clocks
are sampled during the timed loop.  Multi-GPU (torchrun): every rank runs its
own independent batch (weak scaling, no data-path collective); the reported
value is the sum of the work over the max time over ranks.
--impl reference times the fp64 CPU oracle (the only reference this project
has: the pages ship no runnable code) on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    try:
        with open(PEAKS_FILE) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK), "fallback"


def kernel_source_sha(name: str) -> str:
    """Hash of a kernel's sources and of the launch code (api.cu picks the
    grid and the work schedule, which change the DRAM traffic too)."""
    path = os.path.join(ROOT, "attention_forward_13_gb300", "csrc", name)
    h = hashlib.sha256()
    for f in (path, os.path.join(os.path.dirname(path), "ptx.cuh"),
              os.path.join(os.path.dirname(path), "common.cuh"),
              os.path.join(os.path.dirname(path), "api.cu")):
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(workload: str, source: str, scale_units: float = 1.0):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    try:
        with open(TRAFFIC_FILE) as fh:
            d = json.load(fh)
        e = d[workload]
        if e.get("source_sha") != kernel_source_sha(source):
            return None
        return float(e["dram_bytes_per_launch"]) * scale_units
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# work accounting (algorithmic, from the definition; no kernel involvement)
# ---------------------------------------------------------------------------
def causal_pairs(Lq, Lk):
    """Number of (i, j) with j <= i + (Lk - Lq), 0 <= j < Lk, 0 <= i < Lq."""
    tot = 0
    off = Lk - Lq
    for i in range(Lq):
        tot += max(0, min(Lk, i + off + 1))
    return tot


def dense_flops(B, Hq, Lq, Lk, d, causal):
    pairs = causal_pairs(Lq, Lk) if causal else Lq * Lk
    return 4.0 * d * B * Hq * pairs


def window_pairs(Lq, Lk, left, right):
    """Kept (i, j) pairs of a bottom-right band left/right (negative = unbounded)."""
    n = 0
    for i in range(Lq):
        dg = i + Lk - Lq
        lo = 0 if left < 0 else max(0, dg - left)
        hi = Lk - 1 if right < 0 else min(Lk - 1, dg + right)
        n += max(0, hi - lo + 1)
    return n


def varlen_flops(lens, Hq, d, causal):
    return sum(4.0 * d * Hq * (causal_pairs(L, L) if causal else L * L) for L in lens)


def paged_bytes(lens, Hkv, d, Lq, Hq, elem=2):
    kv = sum(lens) * Hkv * d * elem * 2
    qo = 2 * len(lens) * Lq * Hq * d * elem
    return kv + qo + len(lens) * Hq * Lq * 4


# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clocks and throttle reasons during the timed loop."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(work_local: float, ms_local: float, world: int):
    """Whole-job value: total work over all ranks / the slowest rank's time."""
    if world == 1:
        return work_local, ms_local
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([work_local, ms_local], dtype=torch.float64, device=dev)
    w = t[:1].clone()
    m = t[1:].clone()
    dist.all_reduce(w, op=dist.ReduceOp.SUM)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return float(w.item()), float(m.item())


# ---------------------------------------------------------------------------
def time_steps(fn, steps, warmup, stream, flush, passes=1):
    """W untimed steps, then K steps of `passes` passes; before every pass a
    flush, around every pass a pair of events.  Returns the device time of
    each step (the sum of its passes) in ms."""
    import torch
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        step = []
        for _ in range(passes):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            step.append((a, b))
        evs.append(step)
    torch.cuda.synchronize()
    return [sum(a.elapsed_time(b) for a, b in step) for step in evs]


def e2e_pipelined(A, inp, steps, warmup):
    """End-to-end steps of the headline workload through attn_fwd: per step,
    Q, K, V from pinned host memory to the device, the attention, O and LSE
    back to pinned host memory.  Three streams (host-to-device, compute,
    device-to-host) and two device buffer sets; events order step k's
    compute after its inputs arrive and its read-back after its compute, and
    a buffer set is refilled only after the compute that used it.  Returns
    (ms per step from the first input copy to the last read-back, bytes in
    and out per step, ms per step of the same copies alone with both
    directions at once: the host link's bound on a step)."""
    import torch
    host = [t.cpu().pin_memory() for t in (inp.q, inp.k, inp.v)]
    B, Hq, L, _ = inp.q.shape
    h_o = torch.empty(inp.q.shape, dtype=inp.q.dtype).pin_memory()
    h_l = torch.empty((B, Hq, L), dtype=torch.float32).pin_memory()
    dev = [[torch.empty_like(t) for t in (inp.q, inp.k, inp.v)] for _ in range(2)]
    outs = [(torch.empty_like(inp.q), torch.empty((B, Hq, L), dtype=torch.float32, device="cuda"))
            for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def run(n):
        arrived = [torch.cuda.Event() for _ in range(n)]
        computed = [torch.cuda.Event() for _ in range(n)]
        read = [torch.cuda.Event() for _ in range(n)]
        for k in range(n):
            b = k & 1
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(computed[k - 2])  # buffer set b is free again
                for d, h in zip(dev[b], host):
                    d.copy_(h, non_blocking=True)
                arrived[k].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(arrived[k])
                if k >= 2:
                    s_comp.wait_event(read[k - 2])  # outputs b have been read back
                q, kk, v = dev[b]
                A.attn_fwd(q, kk, v, o=outs[b][0], lse=outs[b][1], causal=True, stream=s_comp)
                computed[k].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[k])
                h_o.copy_(outs[b][0], non_blocking=True)
                h_l.copy_(outs[b][1], non_blocking=True)
                read[k].record(s_out)
        return read

    run(warmup)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    read = run(steps)
    end = torch.cuda.Event(enable_timing=True)
    s_out.wait_event(read[-1])
    end.record(s_out)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = h_o.numel() * h_o.element_size() + h_l.numel() * h_l.element_size()

    def copies(n):  # the step's copies without the attention
        for _ in range(n):
            ev = torch.cuda.Event()
            ev.record(s_out)
            s_in.wait_event(ev)
            with torch.cuda.stream(s_in):
                for d, h in zip(dev[0], host):
                    d.copy_(h, non_blocking=True)
            with torch.cuda.stream(s_out):
                h_o.copy_(outs[0][0], non_blocking=True)
                h_l.copy_(outs[0][1], non_blocking=True)
            done = torch.cuda.Event()
            done.record(s_in)
            s_out.wait_event(done)

    copies(2)
    torch.cuda.synchronize()
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record(s_out)
    copies(steps)
    c1.record(s_out)
    torch.cuda.synchronize()
    return ms, h2d, d2h, c0.elapsed_time(c1) / steps


def make_flush():
    import torch
    buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")

    def flush():
        buf.fill_(1.0)
    return flush


def run_ours(args, rank, world, local):
    import torch
    import attention_forward_13_gb300 as A
    from attention_forward_13_gb300 import inputs

    pk, pk_src = peaks()
    stream = torch.cuda.current_stream()
    flush = make_flush()
    dev = "cuda"

    # ---- headline: GQA causal prefill B2 Hq32 Hkv8 L8192 d128 bf16 -----------
    B, Hq, Hkv, L, d = 2, 32, 8, 8192, 128
    inp = inputs.dense(B, Hq, Hkv, L, L, d, "bf16", seed=1003 + 1000 * rank, device=dev,
                       causal=True)
    o = torch.empty_like(inp.q)
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device=dev)
    flops = dense_flops(B, Hq, L, L, d, True)

    def step():
        A.attn_fwd(inp.q, inp.k, inp.v, o=o, lse=lse, causal=True)

    walls = []
    for _ in range(args.warmup):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step()
        torch.cuda.synchronize()
        walls.append(time.perf_counter() - t0)
    # passes per step from the warm-up passes (the first one pays the set-up)
    per = statistics.median(walls[1:] or walls) + 5e-5  # + the flush
    passes = args.passes or max(1, int(math.ceil(args.min_seconds / (per * args.steps))))
    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    wall0 = time.perf_counter()
    times = time_steps(step, args.steps, 0, stream, flush, passes)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    kernel = A.attn_last_kernel_name()
    ms = statistics.mean(times)  # one step = `passes` passes
    total_flops, ms_max = aggregate(flops * passes, ms, world)
    tflops = total_flops / (ms_max * 1e-3) / 1e12
    ms_pass = ms / passes
    kern_tflops = flops / (ms_pass * 1e-3) / 1e12

    # ---- e2e through the public API with host buffers ------------------------
    # Every step copies its Q, K, V from pinned host memory and its O and LSE
    # back.  The copies run on their own streams and overlap the neighbouring
    # steps' attention (double-buffered device inputs and outputs): step k's
    # inputs travel while step k-1 computes, its outputs while step k+1 does.
    e2e_steps = max(3, args.steps // 2)
    e2e_ms, h2d, d2h, link_ms = e2e_pipelined(A, inp, e2e_steps, 2)
    e2e_flops, e2e_ms_max = aggregate(flops, e2e_ms, world)
    _, link_ms_max = aggregate(flops, link_ms, world)
    e2e_value = e2e_flops / (e2e_ms_max * 1e-3) / 1e12
    link_value = e2e_flops / (link_ms_max * 1e-3) / 1e12

    result = {
        "metric": "attn fwd TFLOPS (causal prefill, unmasked pairs) & % of GB300 bf16 tensor peak",
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16)",
        "config": {"workload": "GQA causal prefill B2 Hq32 Hkv8 L8192 d128 bf16 (bottom-right causal)",
                   "B": B, "Hq": Hq, "Hkv": Hkv, "seq_len": L, "head_dim": d, "causal": True,
                   "passes_per_step": passes, "ms_per_pass": round(ms_pass, 4),
                   "parallelism": f"independent batch per GPU x{world}",
                   "l2": "256 MiB buffer written before every pass (flush), outside the events"},
        # The headline kernel runs back to back for the seconds-long timed loop
        # (the GPU reaches its power cap), so its peak is the sustained bf16
        # figure; the burst one is given beside it.
        "roofline": {"bound": "tensor", "achieved": round(kern_tflops, 2),
                     "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                     "frac": round(kern_tflops / pk["bf16_tflops_sustained"], 4),
                     "frac_of_burst_peak": round(kern_tflops / pk["bf16_tflops"], 4),
                     "burst_peak": pk["bf16_tflops"],
                     "traffic": traffic_for("prefill_gqa_B2Hq32Hkv8L8192d128_causal",
                                            "prefill_kernel.cuh"),
                     "peak_source": f"{pk_src} bf16 sustained (MEASURED_PEAKS.json), "
                                    "a 3 s loop at the power cap"
                     if pk_src == "measured" else "fallback 1.7 PFLOP/s sustained",
                     "kernel": kernel,
                     "algorithmic_flops_per_launch": flops},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms_max, 4), "steps": e2e_steps,
                "link_bound": {"ms_per_step": round(link_ms_max, 4), "value": round(link_value, 2),
                               "frac": round(e2e_value / link_value, 4),
                               "gbs": round((h2d + d2h) / (link_ms_max * 1e-3) / 1e9, 1),
                               "note": "the step's copies alone, both directions at once: "
                                       "the host link bounds a step at this"},
                "pipeline": "copies on their own streams, overlapping the neighbouring steps' "
                            "attention (double-buffered device tensors); every step's inputs "
                            "go in and its outputs come out inside the timed region"},
        "gpu_launches": args.steps * passes,
        "clocks": clocks,
        "wall_s_timed_loop": round(wall, 3),
    }
    del inp, o, lse
    torch.cuda.empty_cache()
    if A.attn_device_error() != 0:
        result["device_error"] = True

    if not args.no_extra:
        result["extra"] = run_extra(args, rank, pk, stream, flush)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return result


def run_extra(args, rank, pk, stream, flush, only=None):
    import torch
    import attention_forward_13_gb300 as A
    from attention_forward_13_gb300 import inputs

    steps = max(3, args.steps // 2) if only is None else args.steps
    warm = 3 if only is None else args.warmup
    out = {}
    if only == "gqa":  # the headline workload alone (profiling)
        out.update(_extra_gqa(A, inputs, pk, stream, flush, steps, warm))
    if only in (None, "dense"):
        out.update(_extra_dense(A, inputs, pk, stream, flush, steps, warm))
    if only in (None, "decode"):
        out.update(_extra_decode(A, inputs, pk, stream, flush, steps, warm, args.decode_batch))
    if only in (None, "varlen"):
        out.update(_extra_varlen(A, inputs, pk, stream, flush, steps, warm))
    if only in (None, "masks"):
        out.update(_extra_masks(A, inputs, pk, stream, flush, steps, warm))
    if only in (None, "chunked"):
        out.update(_extra_chunked(A, inputs, pk, stream, flush, steps, warm))
    if only in (None, "fp8"):
        out.update(_extra_fp8(A, inputs, pk, stream, flush, steps, warm))
    return out


def _extra_fp8(A, inputs, pk, stream, flush, steps, warm):
    """FP8 static quantisation on the dense B4 H16 L2048 d128 shape (e4m3
    Q/K/V/O, causal).
    Roofline peak: S = Q K^T runs on the e4m3 tensor path (2x the bf16 rate,
    nominal ratio) and P.V on the fp16 path, half of the FLOPs each, so the
    peak is the measured bf16 peak x 4/3."""
    import torch
    B, H, L, d = 4, 16, 2048, 128
    inp = inputs.dense(B, H, H, L, L, d, "e4m3", seed=1002, device="cuda", causal=True)
    o = torch.empty_like(inp.q)
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    fl = dense_flops(B, H, L, L, d, True)
    t = time_steps(lambda: A.attn_fwd(inp.q, inp.k, inp.v, o=o, lse=lse, causal=True,
                                      scale_p=448.0, scale_o=1.0 / 448.0), steps, warm, stream,
                   flush)
    ms = statistics.mean(t)
    tf = fl / (ms * 1e-3) / 1e12
    peak = pk["bf16_tflops"] * 4.0 / 3.0
    return {"fp8_e4m3_causal_prefill_B4_H16_L2048_d128": {
        "value": round(tf, 2), "unit": "TFLOP/s", "ms": round(ms, 4),
        "kernel": A.attn_last_kernel_name(),
        "roofline": {"bound": "tensor", "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(tf / peak, 4),
                     "peak_note": "measured bf16 x 4/3: S on e4m3 (nominal 2x), P.V on fp16"}}}


def _extra_chunked(A, inputs, pk, stream, flush, steps, warm):
    """Chunked prefill over a paged cache: 8 sequences of U[2048, 8192] cached
    keys (the chunk's own 512 included), Hq 32 / Hkv 8, d 128, page 64, causal."""
    lens = inputs.random_lengths(8, 2048, 8192, seed=1010)
    Lq, Hq, Hkv, d, page = 512, 32, 8, 128, 64
    npages = sum((L + page - 1) // page for L in lens) + 16
    inp = inputs.paged(lens, Lq, Hq, Hkv, d, page, npages, seed=1010, device="cuda", causal=True)
    bt, sl = inp.block_table.cuda(), inp.seqlens_k.cuda()
    fl = sum(4.0 * d * Hq * causal_pairs(Lq, L) for L in lens)
    t = time_steps(lambda: A.attn_fwd_paged(inp.q, inp.k_pool, inp.v_pool, bt, sl, causal=True),
                   steps, warm, stream, flush)
    return {"chunked_prefill_paged_B8_chunk512_Hq32_Hkv8_d128_page64": _tensor_entry(
        fl, statistics.mean(t), pk, A.attn_last_kernel_name())}


def _tensor_entry(fl, ms, pk, kernel, **extra):
    tf = fl / (ms * 1e-3) / 1e12
    e = {"value": round(tf, 2), "unit": "TFLOP/s", "ms": round(ms, 4), "kernel": kernel,
         "roofline": {"bound": "tensor", "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                      "frac": round(tf / pk["bf16_tflops"], 4)}}
    e.update(extra)
    return e


def _extra_masks(A, inputs, pk, stream, flush, steps, warm):
    """The sliding-window, ALiBi and elementwise-bias variants on the dense
    B4 H16 L2048 d128 shape (FLOPs count kept pairs only)."""
    import torch
    out = {}
    B, H, L, d = 4, 16, 2048, 128
    inp = inputs.dense(B, H, H, L, L, d, "bf16", seed=1002, device="cuda", causal=True)
    o = torch.empty_like(inp.q)
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    fl = 4.0 * d * B * H * window_pairs(L, L, 512, 0)
    t = time_steps(lambda: A.attn_fwd(inp.q, inp.k, inp.v, o=o, lse=lse, causal=True,
                                      window=(512, -1)), steps, warm, stream, flush)
    out["window512_causal_prefill_B4_H16_L2048_d128"] = _tensor_entry(
        fl, statistics.mean(t), pk, A.attn_last_kernel_name())
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], device="cuda")
    fl = dense_flops(B, H, L, L, d, True)
    t = time_steps(lambda: A.attn_fwd(inp.q, inp.k, inp.v, o=o, lse=lse, causal=True,
                                      alibi_slopes=slopes), steps, warm, stream, flush)
    out["alibi_causal_prefill_B4_H16_L2048_d128"] = _tensor_entry(
        fl, statistics.mean(t), pk, A.attn_last_kernel_name())
    # One bias per head (bf16 [1,H,L,L], 128 MiB read once per call).
    g = torch.Generator(device="cuda").manual_seed(1009)
    bias = torch.randn((1, H, L, L), generator=g, device="cuda").to(torch.bfloat16)
    q1, k1, v1 = inp.q[:1], inp.k[:1], inp.v[:1]
    o1, l1 = o[:1], lse[:1]
    fl = dense_flops(1, H, L, L, d, False)
    t = time_steps(lambda: A.attn_fwd(q1, k1, v1, o=o1, lse=l1, bias=bias), steps, warm,
                   stream, flush)
    ms = statistics.mean(t)
    out["bias_prefill_B1_H16_L2048_d128"] = _tensor_entry(
        fl, ms, pk, A.attn_last_kernel_name(),
        bias_gbs=round(bias.numel() * 2 / (ms * 1e-3) / 1e9, 1))
    return out


def _extra_dense(A, inputs, pk, stream, flush, steps, warm):
    """Dense causal prefill B4 H16 L2048 d128 bf16."""
    import torch
    B, H, L, d = 4, 16, 2048, 128
    inp = inputs.dense(B, H, H, L, L, d, "bf16", seed=1002, device="cuda", causal=True)
    o = torch.empty_like(inp.q)
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    fl = dense_flops(B, H, L, L, d, True)
    t = time_steps(lambda: A.attn_fwd(inp.q, inp.k, inp.v, o=o, lse=lse, causal=True), steps,
                   warm, stream, flush)
    e = _tensor_entry(fl, statistics.mean(t), pk, A.attn_last_kernel_name())
    e["roofline"]["traffic"] = traffic_for("prefill_B4H16L2048d128_causal", "prefill_kernel.cuh")
    return {"dense_causal_prefill_B4_H16_L2048_d128": e}


def _extra_gqa(A, inputs, pk, stream, flush, steps, warm):
    inp = inputs.workload(3, device="cuda")
    fl = dense_flops(2, 32, 8192, 8192, 128, True)
    t = time_steps(lambda: A.attn_fwd(inp.q, inp.k, inp.v, causal=True), steps, warm, stream,
                   flush)
    ms = statistics.mean(t)
    return {"gqa_causal_prefill_B2_Hq32_Hkv8_L8192_d128": {
        "value": round(fl / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms": round(ms, 4),
        "kernel": A.attn_last_kernel_name(),
        "roofline": {"bound": "tensor", "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(fl / (ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4)}}}


def _extra_decode(A, inputs, pk, stream, flush, steps, warm, batch):
    """Paged decode workload; batch < 64 keeps the first `batch` sequence
    lengths of the workload with a pool of just the pages they need (a smaller
    case for profiling: a few hundred MB on the device).  `value` is the whole
    call (split-KV decode kernel + combine kernel); the combine is also timed
    alone on the same partials, and the decode kernel's own figure is the
    difference."""
    import torch
    B = min(64, batch)
    if B == 64:
        inp = inputs.workload(4, device="cuda")
    else:
        lens_all = inputs.random_lengths(64, 512, 8192, seed=1004)[:B]
        npg = sum((L + 63) // 64 for L in lens_all)
        inp = inputs.paged(lens_all, 1, 32, 8, 128, 64, npg + 16, max_pages=128, seed=1004,
                           device="cuda")
    q = inp.q[:B].contiguous()
    bt, sl = inp.block_table[:B].cuda(), inp.seqlens_k[:B].cuda()
    lens = inp.seqlens_k[:B].tolist()
    nb = paged_bytes(lens, 8, 128, 1, 32)
    splits = A.attn_paged_auto_splits(B, 8, inp.block_table.shape[1])
    rows = B * 32
    ws = torch.empty(max(1, splits * rows * 129), dtype=torch.float32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, 32, 1), dtype=torch.float32, device="cuda")
    t = time_steps(lambda: A.attn_fwd_paged(q, inp.k_pool, inp.v_pool, bt, sl,
                                            num_splits=splits, o=o, lse=lse, workspace=ws),
                   steps, warm, stream, flush)
    kernels = A.attn_last_kernel_name()
    ms = statistics.mean(t)
    gbs = nb / (ms * 1e-3) / 1e9
    key = "paged_decode_B64_Hq32_Hkv8_d128_page64" if B == 64 else f"paged_decode_B{B}_Hq32_Hkv8_d128_page64"
    e = {"value": round(gbs, 1), "unit": "GB/s", "ms": round(ms, 4), "splits": splits,
         "algorithmic_bytes": nb, "kernel": kernels.split("+")[0], "kernels": kernels,
         "roofline": {"bound": "hbm", "peak": pk["hbm_gbs"], "unit": "GB/s",
                      "frac": round(gbs / pk["hbm_gbs"], 4)}}
    if splits > 1:
        op = ws[: splits * rows * 128].view(splits, B, 32, 1, 128)
        lp = ws[splits * rows * 128: splits * rows * 129].view(splits, B, 32, 1)
        tc = time_steps(lambda: A.attn_splitkv_combine(op, lp, o=o, lse=lse), steps, warm,
                        stream, flush)
        ms_c = statistics.mean(tc)
        ms_d = max(ms - ms_c, 1e-6)
        e["combine_ms"] = round(ms_c, 4)
        e["decode_kernel"] = {"ms": round(ms_d, 4), "value": round(nb / (ms_d * 1e-3) / 1e9, 1),
                              "unit": "GB/s", "frac": round(nb / (ms_d * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                              "note": "whole call minus the combine timed alone"}
    return {key: e}


# Special-function throughput of a GB300 SM (results per clock at the 2070 MHz
# nominal clock; an event-timed probe of independent dependency chains):
# ex2.approx 30.2, rcp.approx 15.3 (tanh.approx and lg2 15.3 too).
SFU_PER_CLK = {"ex2": 30.2, "rcp": 15.3}
SFU_CLOCK_HZ = 2.07e9


def softcap_xu_peak_tflops(d, sms=152):
    """Ceiling the special-function unit puts on a soft-capped prefill, in
    TFLOP/s of the usual 4 d FLOP per kept score: each kept score needs two
    ex2 (the tanh's 2^(2y log2 e) and the softmax's) and one rcp (the tanh's
    1 / (e + 1))."""
    sec_per_score = (2.0 / SFU_PER_CLK["ex2"] + 1.0 / SFU_PER_CLK["rcp"]) / (sms * SFU_CLOCK_HZ)
    return 4.0 * d / sec_per_score / 1e12


def _extra_varlen(A, inputs, pk, stream, flush, steps, warm):
    inp = inputs.workload(5, device="cuda")
    cq, ck = inp.cu_seqlens_q.cuda(), inp.cu_seqlens_k.cuda()
    lens = (inp.cu_seqlens_q[1:] - inp.cu_seqlens_q[:-1]).tolist()
    fl = varlen_flops(lens, 16, 64, True)
    t = time_steps(lambda: A.attn_fwd_varlen(inp.q, inp.k, inp.v, cq, ck, inp.max_seqlen_q,
                                             causal=True, softcap=30.0, sink=inp.sink),
                   steps, warm, stream, flush)
    ms = statistics.mean(t)
    return {"varlen_causal_softcap_sink_16seq_H16_d64": {
        "value": round(fl / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms": round(ms, 4),
        "kernel": A.attn_last_kernel_name(),
        "roofline": {"bound": "tensor", "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(fl / (ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4)},
        "roofline_xu": {"bound": "xu", "peak": round(softcap_xu_peak_tflops(64), 1),
                        "unit": "TFLOP/s",
                        "frac": round(fl / (ms * 1e-3) / 1e12 / softcap_xu_peak_tflops(64), 4),
                        "peak_source": "derived: 2 ex2 + 1 rcp per kept score at the special-"
                                       "function rates of this GPU (probe: ex2 30.2, rcp 15.3 "
                                       "results/clk/SM at 2070 MHz, 152 SMs)"}}}


# ---------------------------------------------------------------------------
GQA_L, GQA_D = 8192, 128


def oracle_sample(n_heads, rows, seed=1003):
    """A bounded sample of the GQA causal workload for the fp64 oracle:
    n_heads query heads (4 per kv head) of one batch, each restricted to the
    LAST `rows` of its 8192 query rows against all 8192 keys.  With the
    bottom-right causal mask those rows keep exactly the keys they keep in the
    full problem, so the work per row is the workload's own."""
    from attention_forward_13_gb300 import inputs
    import torch
    hkv = max(1, n_heads // 4)
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((1, n_heads, rows, GQA_D), generator=g).to(torch.bfloat16)
    kv = inputs.dense(1, hkv, hkv, 1, GQA_L, GQA_D, "bf16", seed=seed)
    return [t.to(torch.float64).numpy() for t in (q, kv.k, kv.v)]


def sample_flops(n_heads, rows):
    return 4.0 * GQA_D * n_heads * causal_pairs(rows, GQA_L)


def size_sample(target_seconds, cores):
    """(heads, rows) of a sample the oracle finishes in about target_seconds
    on `cores` threads, from a timed single-head probe of 32 rows."""
    import oracle
    q, k, v = oracle_sample(4, 32)
    t0 = time.perf_counter()  # one (batch, head) problem: one thread does it all
    oracle.attn_dense(q[:, :1], k[:, :1], v[:, :1], 1 / math.sqrt(GQA_D), True)
    per_row = (time.perf_counter() - t0) / 32
    heads = 4 * max(1, (cores + 3) // 4)
    rows = int(target_seconds * cores / (heads * max(per_row, 1e-6)))
    return heads, max(16, min(GQA_L, rows))


def _oracle_threads(cores):
    """The oracle's OpenMP thread count (read once, when its library loads)."""
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))


def cpu_baseline(target_seconds=15.0):
    """Time the fp64 oracle (as it stands) on a bounded sample of the headline
    workload and report the same metric (TFLOP/s on unmasked pairs)."""
    import oracle
    cores = os.cpu_count() or 1
    _oracle_threads(cores)
    heads, rows = size_sample(target_seconds, cores)
    q, k, v = oracle_sample(heads, rows)
    t0 = time.perf_counter()
    oracle.attn_dense(q, k, v, 1 / math.sqrt(GQA_D), True)
    sec = time.perf_counter() - t0
    fl = sample_flops(heads, rows)
    return {"value": round(fl / sec / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{heads} query heads ({heads // 4} kv heads) of the GQA causal "
                      f"workload, the last {rows} of 8192 query rows each against all 8192 "
                      f"keys (d=128), fp64, {sec:.1f} s wall"}


def run_reference(args, rank, world):
    """The oracle timed as the reference arm (rank 0 only): W warm-up steps on
    a tiny sample, then K steps, each the same bounded sample of the headline
    workload (about 5 s of CPU work)."""
    if rank != 0:
        return None
    import oracle
    cores = os.cpu_count() or 1
    _oracle_threads(cores)
    heads, rows = size_sample(5.0, cores)
    q, k, v = oracle_sample(heads, rows)
    fl = sample_flops(heads, rows)
    for _ in range(args.warmup):
        oracle.attn_dense(q[:, :1, :16], k[:, :1], v[:, :1], 1 / math.sqrt(GQA_D), True)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.attn_dense(q, k, v, 1 / math.sqrt(GQA_D), True)
        times.append(time.perf_counter() - t0)
    sec = statistics.mean(times)
    val = fl / sec / 1e12
    sample = (f"{heads} query heads ({heads // 4} kv heads), the last {rows} of 8192 query "
              f"rows each against all 8192 keys, per step; fp64 oracle")
    return {
        "impl": "reference",
        "metric": "attn fwd TFLOPS (causal prefill, unmasked pairs) & % of GB300 bf16 tensor peak",
        "value": round(val, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "GQA causal prefill B2 Hq32 Hkv8 L8192 d128 bf16 (bottom-right causal)",
                   "sample": sample},
        "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--passes", type=int, default=0,
                    help="passes per timed step (0: enough for --min-seconds)")
    ap.add_argument("--min-seconds", type=float, default=3.0)
    ap.add_argument("--only", choices=["gqa", "dense", "decode", "varlen", "masks", "chunked",
                                       "fp8"],
                    default=None,
                    help="run one secondary workload alone (profiling) and print its line")
    ap.add_argument("--decode-batch", type=int, default=64)
    args = ap.parse_args()
    if args.impl == "ours" and args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res))
        return
    rank, world, local = dist_setup(args)
    if args.only is not None:
        import torch
        pk, _ = peaks()
        res = {"only": args.only, "steps": args.steps, "warmup": args.warmup,
               "results": run_extra(args, rank, pk, torch.cuda.current_stream(), make_flush(),
                                    only=args.only)}
        if rank == 0:
            print(json.dumps(res))
        return
    res = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
