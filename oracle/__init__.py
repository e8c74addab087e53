"""fp64 CPU oracle for paged-KV grouped-query decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
bench's ``cpu_baseline`` / ``--impl reference`` legs may import this package.
The CUDA library never imports, links or calls it, and it imports nothing from
the CUDA library.

The arithmetic lives in ``pa_oracle.c`` (plain C, double precision, OpenMP over
(sequence, head)); this module only compiles it with gcc and marshals numpy
arrays.  The definition it follows -- gather K/V rows through the block table,
score with ``scale * q.K``, softmax, weighted sum of V, natural-log LSE -- is
stated in the header comment of ``pa_oracle.c`` with the passages it follows
(paged_attention_v2_pytorch.py commit note, Phase 1 / Phase 2 and GQA
broadcast; apache/tvm PR #20426, section Correctness).

Parity status: pinned (see tests/test_oracle_pins.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into oracle/_build/liboracle.so (gcc -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # No OpenMP runtime: the oracle still works, single-threaded.
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.pa_oracle_decode.argtypes = [i, i, i, i, i, i, i, P, P, P, P, P,
                                     ctypes.c_double, i, P, P, i, i, ctypes.c_double]
    lib.pa_oracle_decode.restype = i
    lib.pa_oracle_scores.argtypes = [i, i, i, i, i, i, P, P, P, P,
                                     ctypes.c_double, i, i, i, P, i, i, ctypes.c_double]
    lib.pa_oracle_scores.restype = i
    lib.pa_oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.pa_oracle_half_to_double.restype = ctypes.c_double
    lib.pa_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.pa_oracle_bf16_to_double.restype = ctypes.c_double
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


DTYPES = {"f16": 0, "bf16": 1, "f32": 2}


def _as_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype in (np.uint16, np.float32):
        return a
    raise TypeError(f"expected float16, bf16 bits (uint16) or float32, got {a.dtype}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
           window: int = 0, num_threads: int = 0, dtype: str = "f16", rope_theta: float = 0.0):
    """fp64 decode attention over a paged KV cache.

    q            float16 [B, Hq, D] (uint16 bf16 bits when dtype="bf16", float32 for "f32")
    k_cache      [num_pages, Hkv, page_size, D] of the same type; v_cache the same
    block_tables int32   [B, max_pages_per_seq]
    context_lens int32   [B]
    rope_theta   > 0: rotate q (position L-1) and K_t (position t) first
    Returns (out float64 [B, Hq, D], lse float64 [B, Hq]).
    """
    lib = _load()
    q = _as_bits(q)
    k = _as_bits(k_cache)
    v = _as_bits(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, Hq, D = q.shape
    num_pages, Hkv, page_size, Dk = k.shape
    if Dk != D or v.shape != k.shape or bt.shape[0] != B or cl.shape != (B,):
        raise ValueError("shape mismatch")
    out = np.empty((B, Hq, D), dtype=np.float64)
    lse = np.empty((B, Hq), dtype=np.float64)
    rc = lib.pa_oracle_decode(B, Hq, Hkv, D, page_size, num_pages, bt.shape[1],
                              _ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(cl),
                              float(scale), int(window), _ptr(out), _ptr(lse),
                              int(num_threads), DTYPES[dtype], float(rope_theta))
    if rc != 0:
        raise OracleError(f"pa_oracle_decode returned {rc}")
    return out, lse


def scores(q, k_cache, block_tables, context_lens, scale: float, window: int,
           b: int, h: int, dtype: str = "f16", rope_theta: float = 0.0) -> np.ndarray:
    """The attended scores scale*q.K_t of one (sequence, head), in fp64."""
    lib = _load()
    q = _as_bits(q)
    k = _as_bits(k_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = k.shape
    cap = int(cl[b])
    s = np.empty(max(cap, 1), dtype=np.float64)
    n = lib.pa_oracle_scores(Hq, Hkv, D, page_size, num_pages, bt.shape[1], _ptr(q),
                             _ptr(k), _ptr(bt), _ptr(cl), float(scale), int(window),
                             int(b), int(h), _ptr(s), cap, DTYPES[dtype], float(rope_theta))
    if n < 0:
        raise OracleError("pa_oracle_scores failed")
    return s[:n].copy()


def half_to_double(bits: int) -> float:
    return _load().pa_oracle_half_to_double(int(bits) & 0xFFFF)


def bf16_to_double(bits: int) -> float:
    return _load().pa_oracle_bf16_to_double(int(bits) & 0xFFFF)
