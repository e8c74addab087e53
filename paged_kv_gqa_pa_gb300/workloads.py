"""Seeded synthetic inputs for paged-KV decode attention.

This module only draws inputs (numpy ``default_rng``; fp32 draws rounded to
fp16 on the host so that every consumer sees identical bits).  It holds none of
the attention arithmetic and imports neither the CUDA library nor the oracle.

Layout of a case (all host numpy arrays):
  q            float16 [B, Hq, D]
  k_cache      float16 [num_pages, Hkv, page_size, D]   (v_cache the same)
  block_tables int32   [B, max_pages_per_seq]   entry j = physical page of the
                                                sequence's logical page j; -1 pads
  context_lens int32   [B]

Page pool recipe: the pool holds sum_b ceil(L_b / page_size) pages plus 25 %
unused slack (or an explicit pool size).  One random permutation of the pool
assigns physical pages to the sequences' logical pages, so the table is
shuffled.  Slack pages are filled with NaN: a gather that strays onto a page no
sequence owns poisons its output.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import math
import os

import numpy as np

PAGE_SIZE = 16


@dataclasses.dataclass
class Case:
    """One decode problem.  dtype "f16" and "f32" arrays hold the values;
    with "bf16", q/k_cache/v_cache hold the uint16 bit patterns of bfloat16
    values (numpy has no bfloat16)."""
    name: str
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    block_tables: np.ndarray
    context_lens: np.ndarray
    scale: float
    window: int
    partition_size: int  # 0 = let the planner choose
    seed: int
    dtype: str = "f16"
    rope_theta: float = 0.0  # > 0: rotary embedding inside the kernel

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def Hq(self):
        return self.q.shape[1]

    @property
    def D(self):
        return self.q.shape[2]

    @property
    def Hkv(self):
        return self.k_cache.shape[1]

    @property
    def page_size(self):
        return self.k_cache.shape[2]

    @property
    def num_pages(self):
        return self.k_cache.shape[0]

    @property
    def max_pages_per_seq(self):
        return self.block_tables.shape[1]

    @property
    def max_context_len(self):
        return int(self.context_lens.max()) if self.context_lens.size else 0


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


BF16_NAN = np.uint16(0x7FC0)


def _fill_normal(out16: np.ndarray, seed_seq: np.random.SeedSequence, std: float,
                 chunk: int = 1 << 24, workers: int | None = None) -> None:
    """Fill a flat 16-bit array with std*N(0,1), drawn in fixed-size chunks, each
    chunk from its own child generator (deterministic for a given seed and size,
    independent of the number of worker threads).  A float16 array gets the
    values rounded to fp16, a float32 array the draws themselves, a uint16
    array bfloat16 bit patterns."""
    flat = out16.reshape(-1)
    n = flat.size
    nchunks = max(1, math.ceil(n / chunk))
    children = seed_seq.spawn(nchunks)

    def work(i):
        lo = i * chunk
        hi = min(n, lo + chunk)
        g = np.random.default_rng(children[i])
        x = g.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        if flat.dtype == np.float16:
            flat[lo:hi] = x.astype(np.float16)
        elif flat.dtype == np.float32:
            flat[lo:hi] = x
        else:
            flat[lo:hi] = to_bf16_bits(x)

    if nchunks == 1:
        work(0)
        return
    workers = workers or min(16, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(work, range(nchunks)))


def make_case(name: str, B: int, Hq: int, Hkv: int, D: int, context_lens, seed: int,
              scale: float | None = None, window: int = 0, q_std: float = 1.0,
              partition_size: int = 0, page_size: int = PAGE_SIZE,
              pool_pages: int | None = None, slack: float = 0.25,
              max_pages_per_seq: int | None = None, nan_slack: bool = True,
              dtype: str = "f16", rope_theta: float = 0.0) -> Case:
    lens = np.asarray(context_lens, dtype=np.int64).reshape(B)
    need = [math.ceil(int(L) / page_size) for L in lens]
    total = int(sum(need))
    if pool_pages is None:
        pool_pages = max(1, total + math.ceil(total * slack))
    if pool_pages < total:
        raise ValueError("page pool smaller than the pages the sequences need")
    maxp = max_pages_per_seq if max_pages_per_seq is not None else max(1, max(need))
    ss = np.random.SeedSequence(seed)
    s_q, s_k, s_v, s_perm = ss.spawn(4)

    et = {"f16": np.float16, "bf16": np.uint16, "f32": np.float32}[dtype]
    q = np.empty((B, Hq, D), dtype=et)
    _fill_normal(q, s_q, q_std)
    k = np.empty((pool_pages, Hkv, page_size, D), dtype=et)
    v = np.empty_like(k)
    _fill_normal(k, s_k, 1.0)
    _fill_normal(v, s_v, 1.0)

    perm = np.random.default_rng(s_perm).permutation(pool_pages).astype(np.int32)
    bt = np.full((B, maxp), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, :need[b]] = perm[off:off + need[b]]
        off += need[b]
    if nan_slack and off < pool_pages:
        slack_ids = perm[off:]
        nan = {"f16": np.float16(np.nan), "bf16": BF16_NAN, "f32": np.float32(np.nan)}[dtype]
        k[slack_ids] = nan
        v[slack_ids] = nan
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return Case(name=name, q=q, k_cache=k, v_cache=v, block_tables=bt,
                context_lens=lens.astype(np.int32), scale=float(scale), window=int(window),
                partition_size=int(partition_size), seed=int(seed), dtype=dtype,
                rope_theta=float(rope_theta))


def _ragged_lengths(B: int, lo: int, hi: int, seed: int, not_multiple_of: int) -> np.ndarray:
    g = np.random.default_rng(np.random.SeedSequence(seed).spawn(5)[4])
    lens = g.integers(lo, hi + 1, size=B)
    lens[0] = 1
    if not np.any(lens % not_multiple_of != 0):
        lens[-1] = hi - 1
    return lens


# The five measured workloads.  Shapes follow the pages' models (Llama-3.2-1B,
# Gemma-2-2b, a 100K-token GQA-6 decode); values are synthetic.
WORKLOADS = {
    "tiny_d64": dict(B=1, Hq=4, Hkv=1, D=64, lens=[256], seed=1001, pool_pages=64),
    "llama3.2-1b_ctx3060": dict(B=1, Hq=32, Hkv=8, D=64, lens=[3060], seed=1002),
    "batch8_ragged_d128": dict(B=8, Hq=32, Hkv=8, D=128, lens="ragged", seed=1003),
    "gemma2-2b_ctx8192_win4096": dict(B=4, Hq=8, Hkv=4, D=256, lens=[8192] * 4, seed=1004,
                                      window=4096, q_std=3.0),
    "gqa6_ctx100k": dict(B=4, Hq=24, Hkv=4, D=256, lens=[100000] * 4, seed=1005,
                         partition_size=512),
}
WORKLOAD_ORDER = list(WORKLOADS)

# Further measured workloads for the widened paths: a bf16 cache at the
# long-context shapes and head_dim 96 (tensor-core kernel only), a rotary
# embedding applied inside the kernel and an fp32 cache (CUDA-core kernel
# only).
EXTRA_WORKLOADS = {
    "gqa6_ctx100k_bf16": dict(B=4, Hq=24, Hkv=4, D=256, lens=[100000] * 4, seed=1006,
                              partition_size=512, dtype="bf16"),
    "gqa4_d96_ctx32k": dict(B=4, Hq=32, Hkv=8, D=96, lens=[32768] * 4, seed=1007),
    # Rotary embedding inside the kernel (Llama-3 frequency base), fp16, D 128.
    "gqa4_rope_ctx32k": dict(B=4, Hq=32, Hkv=8, D=128, lens=[32768] * 4, seed=1008,
                             rope_theta=500000.0),
    # Rotary embedding at head_dim 256 (the long-context GQA-6 shapes, Gemma
    # frequency base 10 000), fp16.
    "gqa6_rope_ctx32k": dict(B=4, Hq=24, Hkv=4, D=256, lens=[32768] * 4, seed=1010,
                             rope_theta=10000.0),
    # An fp32 cache (the dtype the PagedAttention-V2 commit note sizes), D 128.
    "gqa4_f32_ctx32k": dict(B=4, Hq=32, Hkv=8, D=128, lens=[32768] * 4, seed=1009,
                            dtype="f32"),
    # Skewed batches (Llama-3-8B-style heads, 32 query / 8 KV, D 128): one long
    # context among short ones, where a split sized for the longest length
    # leaves most CTAs idle.
    "skewed4_d128_ctx50k": dict(B=4, Hq=32, Hkv=8, D=128, lens=[100, 200, 300, 50000],
                                seed=1011),
    "skewed16_d128_ctx12k": dict(B=16, Hq=32, Hkv=8, D=128, lens=[12000] + [200] * 15,
                                 seed=1012),
    # One sequence of 16K tokens (Llama-3-8B-style heads): a cluster grid of
    # 128 CTAs, fewer than the SMs, which the deep-ring instance serves.
    "single16k_d128": dict(B=1, Hq=32, Hkv=8, D=128, lens=[16384], seed=1013),
}
EXTRA_ORDER = list(EXTRA_WORKLOADS)
ALL_WORKLOADS = {**WORKLOADS, **EXTRA_WORKLOADS}


def workload(name: str, batch: int | None = None) -> Case:
    """One of the measured workloads; `batch` keeps only its first sequences
    (a smaller case of the same shapes, e.g. for profiler captures)."""
    spec = dict(ALL_WORKLOADS[name])
    lens = spec.pop("lens")
    seed = spec["seed"]
    if lens == "ragged":
        lens = _ragged_lengths(spec["B"], 1, 4096, seed, 512)
        spec["max_pages_per_seq"] = 4096 // PAGE_SIZE
    if batch is not None:
        spec["B"] = batch
        lens = list(lens)[:batch]
    return make_case(name=name, B=spec.pop("B"), Hq=spec.pop("Hq"), Hkv=spec.pop("Hkv"),
                     D=spec.pop("D"), context_lens=lens, seed=spec.pop("seed"), **spec)
