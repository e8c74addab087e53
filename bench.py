"""Benchmark of paged-KV GQA decode attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload NAME] [--no-cpu-baseline] [--no-per-workload]

One step = one full decode call (partition kernel + log-sum-exp merge) over
one batch of the workload, inputs resident in HBM.  Rank 0 prints ONE JSON
line.  The metric is KV-read bandwidth: algorithmic bytes = 2 * Hkv * D *
element bytes (one K and one V row) per attended token, divided by the time
per step.

Besides the headline workload, every measured workload gets an entry in
`per_workload` (graph-timed step, single-call time, plan, and the oracle timed
on a bounded sample on the host cores), and the line ends with a compact
`configs` table of the same figures and the pages' own numbers (`context`,
another GPU under WebGPU: context only).

--impl reference times the fp64 CPU oracle on the host cores instead (the only
other path that runs the oracle), on bounded samples of the same workload.
Under torchrun every rank runs its own replica of the workload (weak scaling,
no collective on the data path); time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import glob
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_gqa_pa_gb300 import workloads  # noqa: E402

METRIC = "decode-attn KV-read GB/s (fraction of GB300 HBM peak); µs per decode step"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "gqa6_ctx100k"
PER_WORKLOAD_EAGER_ITERS = 50
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) per launch of the partition kernel, from one ncu
# capture, keyed by workload; valid only while the kernel sources hash to
# `src_sha` (otherwise the bench reports traffic = null).
NCU_TRAFFIC = {
    # One ncu capture of this kernel on the same workload cut to its first
    # sequence (B = 1): (409.72 + 3.71) MB read + written per launch, scaled by
    # tokens to the B = 4 launch.
    ("gqa6_ctx100k", "mma"): {"src_sha": "42f47dba44d6b3c6", "partition_size": 512,
                              "bytes_per_launch": 4 * (409.715712e6 + 3.714304e6)},
}


KERNEL_SOURCES = {
    "mma": ("pa_attend_mma.cuh", "pa_attend_mma_f16.cu", "pa_attend_mma_bf16.cu",
            "pa_attend_mma_rope.cu", "pa_common.cuh"),
    "simt": ("pa_attend.cuh", "pa_attend_d64.cu", "pa_attend_d128.cu", "pa_attend_d256.cu",
             "pa_attend_bf16_d64.cu", "pa_attend_bf16_d128.cu", "pa_attend_bf16_d256.cu",
             "pa_attend_f32_d64.cu", "pa_attend_f32_d128.cu", "pa_attend_f32_d256.cu",
             "pa_common.cuh"),
}


_BLOCK_COMMENT = re.compile(r"/\*.*?\*/", re.S)
_LINE_COMMENT = re.compile(r"//[^\n]*")


def code_only(text: str) -> str:
    """C++/CUDA source without comments, trailing blanks and empty lines, so
    that editing a comment leaves the hash of the code unchanged.  (The
    kernel sources hold no string literal with a comment marker.)"""
    text = _LINE_COMMENT.sub("", _BLOCK_COMMENT.sub("", text))
    return "\n".join(l.rstrip() for l in text.splitlines() if l.strip())


def kernel_src_sha(kernel: str) -> str:
    """Hash of the code (comments stripped) of the sources that define one
    partition-kernel variant."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "paged_kv_gqa_pa_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def attended_tokens(case) -> int:
    n = 0
    for L in case.context_lens.tolist():
        n += min(L, case.window) if case.window > 0 else L
    return n


ELEM_BYTES = {"f16": 2, "bf16": 2, "f32": 4}


def kv_bytes(case) -> int:
    """Algorithmic bytes: one K row and one V row per attended token."""
    return 2 * ELEM_BYTES[case.dtype] * case.Hkv * case.D * attended_tokens(case)


GB300_L2_BYTES = 129 * 10**6  # nominal L2 of one GB300 (the GPU arm asks its device)


def workload_config(case, world: int, l2_bytes: int) -> dict:
    """The `config` of the JSON line: the workload's shapes and how the L2 is
    handled, the same dict for both arms of a run."""
    big = kv_bytes(case) > 2 * l2_bytes
    return {"workload": case.name, "batch": case.B, "num_q_heads": case.Hq,
            "num_kv_heads": case.Hkv, "head_dim": case.D, "page_size": case.page_size,
            "context_lens": "x".join(str(int(x)) for x in sorted(set(case.context_lens.tolist()))),
            "window": case.window, "kv_bytes_per_step": kv_bytes(case),
            "l2": "inputs larger than L2" if big else "L2 flushed between steps",
            "parallelism": f"replicas x{world}"}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.idx = "0"
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.idx = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            if vis:
                self.idx = vis.split(",")[0]
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(ms: float, device, world: int) -> float:
    """The slowest rank's time per step (every rank runs its own replica)."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput_gbs(kv_bytes_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job KV-read GB/s: every rank reads its own replica's bytes each
    step, and the step takes as long as the slowest rank."""
    return kv_bytes_per_rank * world / (ms_per_step * 1e-3) / 1e9


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# The pages' own measurements of this path, quoted as context only: another
# GPU under another API, so nothing here is comparable with the numbers of
# this bench (apache/tvm PR #20426, opening paragraph and section
# Measurements).
PAGES_CONTEXT = {
    "note": "context only; WebGPU, Apple M4 Max; unavailable on this box",
    "sharded_vs_tiled_speedup_3060_tokens": {"D64": 2.95, "D128": 3.89, "D256": 3.49},
    "tiled_kv_read_gbs": 13,
}


def plan_summary(plan):
    """The plan fields that shape a launch, plus a short label."""
    # P<n>: no split; S<tokens> P<partitions> then cl<C> (cluster merge of C
    # CTAs; "d": the deep-ring instance), or x<partitions per CTA> with lc
    # (last-CTA merge) or mk (merge kernel)
    if plan.num_partitions == 1:
        short = "P1"
    elif plan.cluster > 1:
        short = (f"S{plan.partition_size} P{plan.num_partitions} cl{plan.cluster}"
                 + ("d" if plan.deep_ring else ""))
    else:
        short = (f"S{plan.partition_size} P{plan.num_partitions} x{plan.parts_per_cta} "
                 + ("lc" if plan.merge_in_kernel else "mk"))
    return {"partitions": plan.num_partitions, "partition_size": plan.partition_size,
            "ctas": plan.ctas, "cluster": plan.cluster, "merge_in_kernel": plan.merge_in_kernel,
            "parts_per_cta": plan.parts_per_cta, "deep_ring": plan.deep_ring, "short": short}


KERNEL_IDS = {"simt": 1, "mma": 2}
KERNEL_NAMES = {v: k for k, v in KERNEL_IDS.items()}


class GpuArm:
    def __init__(self, case, device, partition_size=None, kernel=None):
        import torch
        import paged_kv_gqa_pa_gb300 as pa
        self.torch = torch
        self.pa = pa
        self.case = case
        self.device = device
        def elems(a):
            t = torch.from_numpy(a)
            return t.view(torch.bfloat16) if case.dtype == "bf16" else t  # f16/f32 as is
        self.q = elems(case.q).to(device)
        self.k = elems(case.k_cache).to(device)
        self.v = elems(case.v_cache).to(device)
        self.bt = torch.from_numpy(case.block_tables).to(device)
        self.cl = torch.from_numpy(case.context_lens).to(device)
        B, Hq, D = case.q.shape
        sms = 0  # plan for the current device, asking it (SM count, clusters per wave)
        ps = case.partition_size if partition_size is None else partition_size
        dtype = {"f16": 0, "bf16": 1, "f32": 2}[case.dtype]
        self.planner_kernel = pa.pa_plan_ex(
            B, Hq, case.Hkv, D, case.page_size, case.num_pages, case.max_pages_per_seq,
            case.max_context_len, case.window, ps, sms, dtype=dtype, kernel=0,
            rope_theta=case.rope_theta).kernel
        self.plan = pa.pa_plan_ex(B, Hq, case.Hkv, D, case.page_size, case.num_pages,
                                  case.max_pages_per_seq, case.max_context_len, case.window, ps,
                                  sms, dtype=dtype, kernel=KERNEL_IDS[kernel] if kernel else 0,
                                  rope_theta=case.rope_theta)
        self.out = torch.empty((B, Hq, D), dtype=self.q.dtype, device=device)
        self.lse = torch.empty((B, Hq), dtype=torch.float32, device=device)
        self.ws = pa.new_workspace(self.plan, device)
        self.stream = torch.cuda.current_stream(device)
        merged_inside = self.plan.cluster > 1 or (
            self.plan.kernel == KERNEL_IDS["mma"] and self.plan.merge_in_kernel)
        self.launches_per_step = 1 if (self.plan.num_partitions == 1 or merged_inside) else 2

    def partitions(self):
        self.pa.pa_decode_partitions(self.plan, self.q, self.k, self.v, self.bt, self.cl,
                                     self.case.scale, self.case.window, self.out, self.lse,
                                     self.ws, self.stream)

    def merge(self):
        self.pa.pa_merge(self.plan, self.cl, self.out, self.lse, self.ws, self.stream)

    def step(self):
        """One decode step through the public call, pa_decode (the partition
        kernel and, where the plan needs it, the merge)."""
        self.pa.pa_decode(self.plan, self.q, self.k, self.v, self.bt, self.cl, self.case.scale,
                          self.case.window, self.out, self.lse, self.ws, self.stream)

    def check_error(self):
        err = self.pa.pa_get_error(self.ws, self.stream)
        if err:
            raise RuntimeError(f"device error word {err:#x}")


def l2_flush_buffer(torch, device):
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    n = max(4 * l2, 1 << 20)
    return torch.ones(n + (-n) % 8, dtype=torch.uint8, device=device)


def time_steps(arm, steps, warmup, graph_steps=50):
    """K decode steps bracketed by two events (inputs larger than L2).  The
    steps are captured once into a CUDA graph of `graph_steps` steps (both
    kernels of each), which is replayed K / graph_steps times -- the way a
    serving loop issues a decode step -- so no host launch gap sits between
    the kernels.  Returns ms per step."""
    torch = arm.torch
    for _ in range(warmup):
        arm.step()
    torch.cuda.synchronize()
    # exactly `steps` steps: the graph holds the largest divisor of K <= graph_steps
    n = max(d for d in range(1, min(graph_steps, steps) + 1) if steps % d == 0)
    reps = steps // n
    stream = torch.cuda.Stream(arm.device)
    saved = arm.stream
    arm.stream = stream
    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                arm.step()
        g.replay()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
        torch.cuda.synchronize()
    arm.stream = saved
    del g
    return start.elapsed_time(end) / (n * reps), n * reps


def time_partition_kernel(arm, steps, flush=None, graph_launches=50):
    """Average duration of one partition-kernel launch, from CUDA events on the
    stream it runs on.

    Inputs larger than L2 (flush is None): `steps` launches of the partition
    kernel alone, captured back to back in a CUDA graph and replayed; the
    events bracket the replays, so the average is the kernel's own time per
    launch with no host launch gap and no merge in between.  Small inputs:
    each launch is bracketed by its own events after an L2 flush (outside the
    events), and the merge runs between launches outside the events."""
    torch = arm.torch
    if flush is None:
        n = max(d for d in range(1, min(graph_launches, steps) + 1) if steps % d == 0)
        reps = steps // n
        stream = torch.cuda.Stream(arm.device)
        saved = arm.stream
        arm.stream = stream
        with torch.cuda.stream(stream):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(n):
                    arm.partitions()
            g.replay()
            torch.cuda.synchronize()
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            for _ in range(reps):
                g.replay()
            end.record(stream)
            torch.cuda.synchronize()
        arm.stream = saved
        del g
        # the graph's last launch leaves partials unmerged: finish that step
        arm.merge()
        torch.cuda.synchronize()
        return start.elapsed_time(end) / (n * reps), "CUDA graph of back-to-back launches"
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush_l2(flush)
        ev[i][0].record(arm.stream)
        arm.partitions()
        ev[i][1].record(arm.stream)
        arm.merge()
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev), "per-launch events, L2 flushed"


def flush_l2(flush):
    """Evict L2 by READING a buffer larger than it (a sum on the device): the
    lines it leaves are clean, so the next kernel's reads do not pay for
    writing the flush back."""
    import torch
    return flush.view(torch.int64).sum()


def time_flushed(arm, iters, flush, reps=3):
    """Single-call time from a cold L2.  `iters` pairs of (an L2 eviction by
    reading a buffer larger than it, one pa_decode call) run back to back
    between two events, and so do `iters` evictions alone; the difference
    per pair is the call's cost on the stream: its launch behind a kernel
    that does not launch dependents early, its run from a cold L2, and none
    of the overlap with a preceding step that back-to-back steps get.  No
    host time is inside (the device never waits for the host: an eviction
    takes far longer than enqueueing a call).  A difference of two long
    intervals also averages out the CUDA events' ~2 us granularity.
    Returns (ms per call, the median of `reps` such differences; median host
    microseconds spent inside one pa_decode call)."""
    torch = arm.torch
    for _ in range(3):
        arm.step()
    torch.cuda.synchronize()
    host = []

    def run(with_call):
        a, b = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        flush_l2(flush)
        a.record(arm.stream)
        for _ in range(iters):
            flush_l2(flush)
            if with_call:
                t0 = time.perf_counter()
                arm.step()
                host.append((time.perf_counter() - t0) * 1e6)
        b.record(arm.stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    diffs = []
    for _ in range(reps):
        t_flush = run(False)
        t_both = run(True)
        diffs.append((t_both - t_flush) / iters)
    return statistics.median(diffs), statistics.median(host)


def time_isolated(arm, iters, flush):
    """One call bracketed by its own pair of CUDA events, per iteration, after
    an L2 eviction (events and call enqueued behind the eviction): median ms.
    The start event keeps the call from starting early behind the eviction
    kernel, and the events tick in ~2 us steps."""
    torch = arm.torch
    res = []
    for _ in range(iters):
        flush_l2(flush)
        a, b = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        a.record(arm.stream)
        arm.step()
        b.record(arm.stream)
        torch.cuda.synchronize()
        res.append(a.elapsed_time(b))
    return statistics.median(res)


def host_us_prepared(arm, calls=200):
    """Host microseconds per launch through a prepared pa_decode (arguments
    checked once; the C call alone per step), averaged over `calls` calls
    issued back to back."""
    torch = arm.torch
    call = arm.pa.prepare_decode(arm.plan, arm.q, arm.k, arm.v, arm.bt, arm.cl, arm.case.scale,
                                 arm.case.window, arm.out, arm.lse, arm.ws, arm.stream)
    call()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(calls):
        call()
    t1 = time.perf_counter()
    torch.cuda.synchronize()
    return (t1 - t0) * 1e6 / calls


def time_graph_rotating(case, device, kernel, min_steps=40, max_copies=64,
                        max_bytes=4 << 30, partition_size=None):
    """Steps captured in one CUDA graph, cycling over C copies of the K/V pools so
    that each step reads data the previous C-1 steps have evicted from L2 (C is
    chosen so the copies together exceed 3x L2, within max_copies/max_bytes).
    Returns (us per step, us of the partition kernel alone, copies, L2 state)."""
    import torch
    arm = GpuArm(case, device, kernel=kernel, partition_size=partition_size)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    pool = arm.k.numel() * arm.k.element_size() * 2  # K and V
    C = max(1, min(max_copies, math.ceil(3 * l2 / max(pool, 1)), max(1, max_bytes // pool)))
    ks = [arm.k] + [arm.k.clone() for _ in range(C - 1)]
    vs = [arm.v] + [arm.v.clone() for _ in range(C - 1)]
    cold = C * pool > 2 * l2
    n = max(min_steps, C)
    n = C * math.ceil(n / C)
    stream = torch.cuda.Stream(device)

    def run(i, merge=True):
        arm.k, arm.v = ks[i % C], vs[i % C]
        arm.stream = stream
        arm.partitions()
        if merge:
            arm.merge()

    res = []
    for merge in (True, False):
        with torch.cuda.stream(stream):
            for i in range(C):
                run(i, merge)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    run(i, merge)
            g.replay()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(3):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
        res.append(a.elapsed_time(b) * 1e3 / (3 * n))
        del g
    arm.stream = torch.cuda.current_stream(device)
    arm.check_error()
    out = (res[0], res[1], C, "cold (rotating copies)" if cold else "warm (fits in L2)", arm.plan)
    del ks, vs, arm
    torch.cuda.empty_cache()
    return out


def e2e_steps(arm, steps, warmup, upload_kv=False, pipelined=True):
    """Through the public API with host buffers: per step, copy the step's inputs
    (q, block table, context lengths; with upload_kv also the K/V pools) from
    pinned host memory, decode, and read out + LSE back to pinned host memory.

    pipelined: the way a serving loop runs it -- two sets of per-step device
    and host buffers, the input copies on one stream, the decode on the
    compute stream, the result copies on a third, ordered by events, so that
    step i+1's inputs and step i-1's results move while step i computes.
    Otherwise every copy and the decode run in order on one stream.
    Returns (ms per step, H2D bytes per step, D2H bytes per step)."""
    torch = arm.torch
    c = arm.case
    dev = arm.device

    def host(a):
        t = torch.from_numpy(a)
        return (t.view(torch.bfloat16) if c.dtype == "bf16" else t).pin_memory()

    nbuf = 2 if pipelined else 1
    hq = [host(c.q) for _ in range(nbuf)]
    hbt = [torch.from_numpy(c.block_tables).pin_memory() for _ in range(nbuf)]
    hcl = [torch.from_numpy(c.context_lens).pin_memory() for _ in range(nbuf)]
    hout = [torch.empty(arm.out.shape, dtype=arm.out.dtype).pin_memory() for _ in range(nbuf)]
    hlse = [torch.empty(arm.lse.shape, dtype=arm.lse.dtype).pin_memory() for _ in range(nbuf)]
    dq = [arm.q] + [torch.empty_like(arm.q) for _ in range(nbuf - 1)]
    dbt = [arm.bt] + [torch.empty_like(arm.bt) for _ in range(nbuf - 1)]
    dcl = [arm.cl] + [torch.empty_like(arm.cl) for _ in range(nbuf - 1)]
    dout = [arm.out] + [torch.empty_like(arm.out) for _ in range(nbuf - 1)]
    dlse = [arm.lse] + [torch.empty_like(arm.lse) for _ in range(nbuf - 1)]
    hk = hv = None
    if upload_kv:
        hk = host(c.k_cache)
        hv = host(c.v_cache)
    h2d = hq[0].numel() * hq[0].element_size() + hbt[0].numel() * 4 + hcl[0].numel() * 4
    if upload_kv:
        h2d += hk.numel() * hk.element_size() + hv.numel() * hv.element_size()
    d2h = hout[0].numel() * hout[0].element_size() + hlse[0].numel() * 4

    comp = arm.stream
    s_in = torch.cuda.Stream(dev) if pipelined else comp
    s_out = torch.cuda.Stream(dev) if pipelined else comp
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_done = [torch.cuda.Event() for _ in range(nbuf)]
    ev_read = [torch.cuda.Event() for _ in range(nbuf)]
    saved = (arm.q, arm.bt, arm.cl, arm.out, arm.lse)

    def one(i):
        j = i % nbuf
        with torch.cuda.stream(s_in):
            if i >= nbuf:
                s_in.wait_event(ev_done[j])   # buffer set j's previous decode is done
            dq[j].copy_(hq[j], non_blocking=True)
            dbt[j].copy_(hbt[j], non_blocking=True)
            dcl[j].copy_(hcl[j], non_blocking=True)
            if upload_kv:
                arm.k.copy_(hk, non_blocking=True)
                arm.v.copy_(hv, non_blocking=True)
            ev_in[j].record(s_in)
        comp.wait_event(ev_in[j])
        if i >= nbuf:
            comp.wait_event(ev_read[j])       # its previous results have been read
        arm.q, arm.bt, arm.cl, arm.out, arm.lse = dq[j], dbt[j], dcl[j], dout[j], dlse[j]
        arm.step()
        ev_done[j].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[j])
            hout[j].copy_(dout[j], non_blocking=True)
            hlse[j].copy_(dlse[j], non_blocking=True)
            ev_read[j].record(s_out)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(steps):
        one(warmup + i)
    # the end: every stream's work of the timed steps
    comp.wait_stream(s_in)
    comp.wait_stream(s_out)
    b.record(comp)
    torch.cuda.synchronize()
    arm.q, arm.bt, arm.cl, arm.out, arm.lse = saved
    ms = a.elapsed_time(b) / steps
    return ms, h2d, d2h


class OracleSampler:
    """Times the oracle, as it stands, on a bounded sample of the workload.

    The sample is the whole decode step (every sequence and head), repeated
    as often as the time budget allows, when one step fits the budget;
    otherwise sequence 0 with all its query heads over the last L of its
    attended tokens, L sized to the budget.  The per-token cost comes from a
    one-thread calibration run."""

    def __init__(self, case, threads=0):
        import oracle
        self.oracle = oracle
        self.case = case
        self.threads = threads or os.cpu_count() or 1
        L0 = int(case.context_lens[0])
        self.att = min(L0, case.window) if case.window > 0 else L0
        self.total = attended_tokens(case)
        probe = max(1, min(self.att, 512))
        t0 = time.perf_counter()
        self._run(self._sub(probe), 1)
        # seconds per (attended token, query head) on one thread
        self.sec_per_unit_1thread = max((time.perf_counter() - t0) / (probe * case.Hq), 1e-12)

    def _sub(self, L):
        c = self.case
        return workloads.Case(name=c.name + "_sample", q=np.ascontiguousarray(c.q[:1]),
                              k_cache=c.k_cache, v_cache=c.v_cache,
                              block_tables=c.block_tables[:1],
                              context_lens=c.context_lens[:1].copy(), scale=c.scale, window=L,
                              partition_size=0, seed=c.seed, dtype=c.dtype,
                              rope_theta=c.rope_theta)

    def _run(self, s, threads):
        self.oracle.decode(s.q, s.k_cache, s.v_cache, s.block_tables, s.context_lens, s.scale,
                           s.window, num_threads=threads, dtype=s.dtype,
                           rope_theta=s.rope_theta)

    def plan(self, budget_s):
        """(repeats of the whole step, or 0) and L for a sample of about budget_s."""
        c = self.case
        full_s = self.sec_per_unit_1thread * self.total * c.Hq / min(self.threads, c.B * c.Hq)
        if full_s <= budget_s:
            return max(1, int(budget_s / max(full_s, 1e-9))), self.total
        L = int(budget_s * min(self.threads, c.Hq) / (self.sec_per_unit_1thread * c.Hq))
        return 0, max(16, min(self.att, L))

    def run(self, sample):
        """Time one sample from plan(); returns (GB/s, seconds, description, threads)."""
        reps, L = sample
        c = self.case
        t0 = time.perf_counter()
        if reps:
            for _ in range(reps):
                self._run(c, self.threads)
            tokens = reps * self.total
            used = min(self.threads, c.B * c.Hq)
            desc = (f"the whole step ({c.B} sequences x {c.Hq} query heads, {self.total} "
                    f"attended tokens) run {reps} times; fp64 C oracle, OpenMP over "
                    f"(sequence, head)")
        else:
            self._run(self._sub(L), self.threads)
            tokens = L
            used = min(self.threads, c.Hq)
            desc = (f"sequence 0 of {c.B}, all {c.Hq} query heads, last {L} of {self.att} "
                    f"attended tokens; fp64 C oracle, OpenMP over heads")
        dt = time.perf_counter() - t0
        byts = 2 * ELEM_BYTES[c.dtype] * c.Hkv * c.D * tokens
        return byts / dt / 1e9, dt, desc, used

    def single_thread_gbs(self):
        """The oracle on one thread, from the calibration run: KV GB/s."""
        c = self.case
        per_token = self.sec_per_unit_1thread * c.Hq  # seconds per attended token, all heads
        return 2 * ELEM_BYTES[c.dtype] * c.Hkv * c.D / per_token / 1e9


def run_reference(args):
    world, rank, local = dist_setup()
    if rank != 0:
        return 0
    case = workloads.workload(args.workload)
    sampler = OracleSampler(case)
    per_step_budget = args.reference_budget_s / max(1, args.steps + args.warmup)
    sample = sampler.plan(per_step_budget)
    for _ in range(args.warmup):
        sampler.run(sample)
    vals, secs = [], []
    desc, used = "", 1
    for _ in range(args.steps):
        v, dt, desc, used = sampler.run(sample)
        vals.append(v)
        secs.append(dt)
    value = statistics.median(vals)
    line = {
        # n_gpus: the launch's N, as on the other arm's line; this arm runs on
        # rank 0's host cores only (config.device, cpu_baseline.cores)
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.median(secs) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(case, world, GB300_L2_BYTES),
        "device": "host CPU (oracle)",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": desc, "single_thread_value": sampler.single_thread_gbs()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    import torch
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    case = workloads.workload(args.workload, batch=args.batch)
    arm = GpuArm(case, device, kernel=None if args.kernel == "auto" else args.kernel)
    byts = kv_bytes(case)
    flush = None
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    big = byts > 2 * l2
    if not big:
        flush = l2_flush_buffer(torch, device)

    # correctness of the launch configuration being timed (device error word)
    arm.step()
    arm.check_error()
    if args.profile_only:
        # A short, plain run for ncu: warm-up plus `steps` decode steps, no
        # timing, sampling or baselines.
        for _ in range(args.warmup + args.steps):
            arm.step()
        torch.cuda.synchronize()
        arm.check_error()
        if rank == 0:
            print(json.dumps({"profile_only": True, "workload": args.workload,
                              "steps": args.steps, "warmup": args.warmup,
                              "partitions": arm.plan.num_partitions,
                              "partition_size": arm.plan.partition_size}), flush=True)
        return 0

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(device) as clk:
        if big:
            ms, timed_steps = time_steps(arm, args.steps, args.warmup)
        else:
            ms, _ = time_flushed(arm, args.steps, flush, reps=1)  # exactly K timed steps
            timed_steps = args.steps
        kern_ms, kern_timing = time_partition_kernel(arm, min(args.steps, 500), flush)
    if world > 1:
        torch.distributed.barrier()
    arm.check_error()
    ms_max = max_over_ranks(ms, device, world)
    value = job_throughput_gbs(byts, world, ms_max)

    peak, peak_kind = measured_peaks()
    kern_gbs = byts / (kern_ms * 1e-3) / 1e9
    kname = KERNEL_NAMES[arm.plan.kernel]
    sha = kernel_src_sha(kname)
    tr = NCU_TRAFFIC.get((args.workload, kname))
    traffic = None
    if tr and tr["src_sha"] == sha and tr["partition_size"] == arm.plan.partition_size \
            and args.batch is None:
        traffic = tr["bytes_per_launch"]

    e2e_ms, h2d, d2h = e2e_steps(arm, max(10, min(args.steps, 200)), 3)
    ser_ms, _, _ = e2e_steps(arm, max(10, min(args.steps, 200)), 3, pipelined=False)
    e2e = {"value": byts / (e2e_ms * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "note": "per step: H2D of q, block table, context lengths (KV cache resident); "
                   "pa_decode; D2H of out and LSE -- pipelined over two buffer sets and three "
                   "streams as a serving loop runs it",
           "serial": {"value": byts / (ser_ms * 1e-3) / 1e9, "ms_per_step": ser_ms,
                      "note": "the same with every copy and the decode in order on one stream"}}
    e2e_kv = None
    if not args.no_kv_upload:
        kv_ms, kv_h2d, kv_d2h = e2e_steps(arm, 5, 1, upload_kv=True, pipelined=False)
        e2e_kv = {"value": byts / (kv_ms * 1e-3) / 1e9, "unit": UNIT,
                  "h2d_bytes_per_step": kv_h2d, "d2h_bytes_per_step": kv_d2h,
                  "ms_per_step": kv_ms}
    arm.check_error()

    per = None
    summary = summary_extra = None
    if not args.no_per_workload and rank == 0:
        per = {}
        # One compact row per workload: the five named configs early in the
        # line ("configs"), the further workloads at its end ("configs_extra").
        fields = ["us/step", "KV GB/s", "frac measured HBM", "frac nominal 8 TB/s",
                  "single-call us", "oracle GB/s", "plan"]
        summary = {"fields": fields, "oracle_cores": None}
        summary_extra = {"fields": ["kernel"] + fields}
        wl_flush = flush if flush is not None else l2_flush_buffer(torch, device)
        for name in workloads.WORKLOAD_ORDER + workloads.EXTRA_ORDER:
            c = case if name == args.workload else workloads.workload(name)
            b = kv_bytes(c)
            entry = {"dtype": c.dtype, "head_dim": c.D, "rope_theta": c.rope_theta}
            simt_ok = c.D in (64, 128, 256)
            kernels = ("mma", "simt") if simt_ok else ("mma",)
            if c.dtype == "f32":
                kernels = ("simt",)  # no tensor-core build for fp32 caches
            for kname in kernels:
                us, kus, copies, l2state, plan = time_graph_rotating(c, device, kname)
                # single calls from a cold L2, each behind a kernel that does
                # not launch dependents early; then the same plan without the
                # pre-wait prefetch, which such a caller would choose
                earm = GpuArm(c, device, kernel=kname)
                eager_ms, host_us = time_flushed(earm, args.per_workload_iters, wl_flush)
                iso_ms = time_isolated(earm, args.per_workload_iters, wl_flush)
                prep_us = host_us_prepared(earm)
                earm.plan.prewait_prefetch = 0
                eager0_ms, _ = time_flushed(earm, args.per_workload_iters, wl_flush)
                earm.check_error()
                del earm
                entry[kname] = {"us_per_step": us, "partition_kernel_us": kus,
                                "kv_gbs": b / (us * 1e-6) / 1e9,
                                "single_call_us": eager_ms * 1e3,
                                "single_call_kv_gbs": b / (eager_ms * 1e-3) / 1e9,
                                "single_call_us_no_prewait": eager0_ms * 1e3,
                                "single_call_isolated_us": iso_ms * 1e3,
                                "host_us_in_pa_decode": host_us,
                                "host_us_prepared_call": prep_us,
                                "frac_of_measured_hbm": b / (us * 1e-6) / 1e9 / peak,
                                "frac_of_nominal_8tbs": b / (us * 1e-6) / 1e9 / NOMINAL_HBM_GBS,
                                "plan": plan_summary(plan)}
                entry.update({"copies": copies, "l2": l2state})
            oracle_cpu = None
            if not args.no_cpu_baseline:
                # the oracle beside each workload: a bounded sample on the host cores
                sampler = OracleSampler(c)
                v, dt, desc, used = sampler.run(sampler.plan(args.per_workload_cpu_budget_s))
                oracle_cpu = {"value": v, "unit": UNIT, "cores": used, "kind": "oracle",
                              "sample": desc, "seconds": dt,
                              "single_thread_value": sampler.single_thread_gbs()}
            entry.update({"kv_bytes": b, "cpu_baseline": oracle_cpu,
                          "timing": "us_per_step: CUDA graph of back-to-back steps over "
                                    "rotating K/V copies; single_call_us: "
                                    f"{args.per_workload_iters} (L2 eviction by reading, one "
                                    "pa_decode call) pairs back to back minus the evictions "
                                    "alone, per call (median of 3), CUDA events on the stream; "
                                    "_no_prewait: the same plan with prewait_prefetch 0; "
                                    "single_call_isolated_us: median of one call between its "
                                    "own event pair after each eviction"})
            per[name] = entry
            k0 = kernels[0]
            e0 = entry[k0]
            row = [round(e0["us_per_step"], 2), round(e0["kv_gbs"]),
                   round(e0["frac_of_measured_hbm"], 3), round(e0["frac_of_nominal_8tbs"], 3),
                   round(e0["single_call_us"], 1),
                   round(oracle_cpu["value"], 3) if oracle_cpu else None,
                   e0["plan"]["short"]]
            if name in workloads.WORKLOAD_ORDER:
                summary[name] = row
                if oracle_cpu:
                    summary["oracle_cores"] = oracle_cpu["cores"]
            else:
                summary_extra[name] = [k0] + row

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        sampler = OracleSampler(case)
        v, dt, desc, used = sampler.run(sampler.plan(args.cpu_budget_s))
        cpu = {"value": v, "unit": UNIT, "cores": used, "kind": "oracle", "sample": desc,
               "seconds": dt, "single_thread_value": sampler.single_thread_gbs()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "us_per_step": ms_max * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": case.dtype,
            "data": "synthetic",
            "config": workload_config(case, world, l2),
            # Early, so that a record keeping only the head of the line has
            # them: each named config's figures beside the oracle's, and the
            # pages' own figures (context only).
            "configs": summary,
            "context": PAGES_CONTEXT,
            "plan": plan_summary(arm.plan),
            "roofline": {"bound": "hbm", "achieved": kern_gbs, "peak": peak, "unit": "GB/s",
                         "frac": kern_gbs / peak, "traffic": traffic,
                         "peak_kind": peak_kind,
                         "kernel": f"partition kernel ({KERNEL_NAMES[arm.plan.kernel]})",
                         "kernel_us": kern_ms * 1e3, "kernel_timing": kern_timing,
                         "frac_of_nominal_8tbs":
                             kern_gbs / NOMINAL_HBM_GBS, "src_sha": sha},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "e2e_with_kv_upload": e2e_kv,
            "gpu_launches": timed_steps * arm.launches_per_step,
            "timed_loop": "CUDA graph replays of captured steps" if big else
                          "per-step launches, L2 flushed between steps",
            "clocks": clk.summary(),
            "per_workload": per,
            "configs_extra": summary_extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=workloads.WORKLOAD_ORDER + workloads.EXTRA_ORDER)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--no-kv-upload", action="store_true")
    ap.add_argument("--kernel", default="auto", choices=["auto", "mma", "simt"])
    ap.add_argument("--batch", type=int, default=None,
                    help="keep only the workload's first sequences (profiler captures)")
    ap.add_argument("--profile-only", action="store_true",
                    help="run warm-up + steps untimed (for ncu captures) and exit")
    ap.add_argument("--per-workload-iters", type=int, default=PER_WORKLOAD_EAGER_ITERS)
    ap.add_argument("--per-workload-cpu-budget-s", type=float, default=2.0)
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
