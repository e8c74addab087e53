"""ctypes binding of libpa_gb300.so (include/pa.h), argument marshalling only.

Every function here checks and converts arguments (torch CUDA tensors ->
device pointers, the current torch stream -> cudaStream_t) and calls the C ABI
of the same name; all computation runs in the library's CUDA kernels.  There
is no CPU fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_CUDA = 3
PA_ERR_WORKSPACE = 4
PA_DEVERR_BAD_PAGE = 1
PA_DEVERR_BAD_LENGTH = 2
PA_DEVERR_TIMEOUT = 4
PA_KERNEL_SIMT = 1
PA_KERNEL_MMA = 2
PA_DTYPE_F16 = 0
PA_DTYPE_BF16 = 1
PA_DTYPE_F32 = 2
PA_PARTITION_BALANCED = -1
_TORCH_DTYPE = {PA_DTYPE_F16: torch.float16, PA_DTYPE_BF16: torch.bfloat16,
                PA_DTYPE_F32: torch.float32}

EXPORTED = ("pa_plan", "pa_plan_ex", "pa_decode", "pa_decode_partitions", "pa_merge",
            "pa_get_error", "pa_get_error_ex", "pa_status_string", "pa_version",
            "pa_decode_static")


class pa_plan_t(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("num_q_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("num_pages", ctypes.c_int),
        ("max_pages_per_seq", ctypes.c_int),
        ("max_context_len", ctypes.c_int),
        ("window", ctypes.c_int),
        ("partition_size", ctypes.c_int),
        ("num_partitions", ctypes.c_int),
        ("heads_per_cta", ctypes.c_int),
        ("num_sms", ctypes.c_int),
        ("ctas", ctypes.c_int),
        ("workspace_bytes", ctypes.c_size_t),
        ("kernel", ctypes.c_int),
        ("parts_per_cta", ctypes.c_int),
        ("merge_in_kernel", ctypes.c_int),
        ("ctrl_bytes", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("rope_theta", ctypes.c_float),
        ("cluster", ctypes.c_int),
        ("prewait_prefetch", ctypes.c_int),
        ("test_stall_bytes", ctypes.c_int),
        ("balanced", ctypes.c_int),
        ("deep_ring", ctypes.c_int),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class PAError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} failed: {status} ({pa_status_string(status)})")
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Load the built library (built by paged_kv_gqa_pa_gb300.build / __graft_entry__.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is not built; run `python -m paged_kv_gqa_pa_gb300.build` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i = ctypes.c_int
        pp = ctypes.POINTER(pa_plan_t)
        lib.pa_plan.argtypes = [i] * 11 + [pp]
        lib.pa_plan.restype = i
        lib.pa_plan_ex.argtypes = [i] * 13 + [ctypes.c_float, pp]
        lib.pa_plan_ex.restype = i
        dec = [pp, P, P, P, P, P, ctypes.c_float, i, P, P, P, P]
        lib.pa_decode.argtypes = dec
        lib.pa_decode.restype = i
        lib.pa_decode_partitions.argtypes = dec
        lib.pa_decode_partitions.restype = i
        lib.pa_merge.argtypes = [pp, P, P, P, P, P]
        lib.pa_merge.restype = i
        lib.pa_get_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_int)]
        lib.pa_get_error.restype = i
        lib.pa_get_error_ex.argtypes = [P, P, i, ctypes.POINTER(ctypes.c_uint)]
        lib.pa_get_error_ex.restype = i
        lib.pa_status_string.argtypes = [i]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_version.argtypes = []
        lib.pa_version.restype = i
        lib.pa_decode_static.argtypes = dec[:10] + [P]
        lib.pa_decode_static.restype = i
        _lib = lib
        return lib


def pa_status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def pa_version() -> int:
    return load().pa_version()


def pa_plan(batch, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
            max_pages_per_seq, max_context_len, window=0, partition_size=0,
            num_sms=0) -> pa_plan_t:
    plan = pa_plan_t()
    st = load().pa_plan(int(batch), int(num_q_heads), int(num_kv_heads), int(head_dim),
                        int(page_size), int(num_pages), int(max_pages_per_seq),
                        int(max_context_len), int(window), int(partition_size), int(num_sms),
                        ctypes.byref(plan))
    if st != PA_OK:
        raise PAError("pa_plan", st)
    return plan


def pa_plan_ex(batch, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
               max_pages_per_seq, max_context_len, window=0, partition_size=0, num_sms=0,
               dtype=PA_DTYPE_F16, kernel=0, rope_theta=0.0) -> pa_plan_t:
    plan = pa_plan_t()
    st = load().pa_plan_ex(int(batch), int(num_q_heads), int(num_kv_heads), int(head_dim),
                           int(page_size), int(num_pages), int(max_pages_per_seq),
                           int(max_context_len), int(window), int(partition_size), int(num_sms),
                           int(dtype), int(kernel), ctypes.c_float(rope_theta),
                           ctypes.byref(plan))
    if st != PA_OK:
        raise PAError("pa_plan_ex", st)
    return plan


def _dev_ptr(t, name, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _decode_args(plan, q, k_cache, v_cache, block_tables, context_lens, scale, window, out, lse,
                 workspace, stream):
    et = _TORCH_DTYPE.get(plan.dtype, torch.float16)
    return (ctypes.byref(plan), _dev_ptr(q, "q", et),
            _dev_ptr(k_cache, "k_cache", et),
            _dev_ptr(v_cache, "v_cache", et),
            _dev_ptr(block_tables, "block_tables", torch.int32),
            _dev_ptr(context_lens, "context_lens", torch.int32), ctypes.c_float(scale),
            int(window), _dev_ptr(out, "out", et), _dev_ptr(lse, "lse", torch.float32),
            _dev_ptr(workspace, "workspace"), _stream_ptr(stream))


def pa_decode(plan, q, k_cache, v_cache, block_tables, context_lens, scale, window, out, lse,
              workspace, stream=None) -> None:
    st = load().pa_decode(*_decode_args(plan, q, k_cache, v_cache, block_tables, context_lens,
                                        scale, window, out, lse, workspace, stream))
    if st != PA_OK:
        raise PAError("pa_decode", st)


class PreparedDecode:
    """pa_decode with its arguments checked and converted once.

    A decode loop calls pa_decode with the same buffers every step (their
    contents change, their addresses do not).  This object keeps the checked
    ctypes arguments and the plan, so each call is the C call alone: a few
    microseconds of host time instead of the per-tensor checks of pa_decode.
    The tensors must stay alive and in place while it is used."""

    def __init__(self, plan, q, k_cache, v_cache, block_tables, context_lens, scale, window, out,
                 lse, workspace, stream=None):
        self.plan = pa_plan_t.from_buffer_copy(plan)  # the plan as it was when prepared
        self._keep = (q, k_cache, v_cache, block_tables, context_lens, out, lse, workspace)
        args = _decode_args(self.plan, q, k_cache, v_cache, block_tables, context_lens, scale,
                            window, out, lse, workspace, stream)
        self._fn = load().pa_decode
        self._args = args

    def __call__(self) -> None:
        st = self._fn(*self._args)
        if st != PA_OK:
            raise PAError("pa_decode", st)


def prepare_decode(plan, q, k_cache, v_cache, block_tables, context_lens, scale, window, out, lse,
                   workspace, stream=None) -> PreparedDecode:
    """Check and convert pa_decode's arguments once; calling the result launches."""
    return PreparedDecode(plan, q, k_cache, v_cache, block_tables, context_lens, scale, window,
                          out, lse, workspace, stream)


def pa_decode_partitions(plan, q, k_cache, v_cache, block_tables, context_lens, scale, window,
                         out, lse, workspace, stream=None) -> None:
    st = load().pa_decode_partitions(*_decode_args(plan, q, k_cache, v_cache, block_tables,
                                                   context_lens, scale, window, out, lse,
                                                   workspace, stream))
    if st != PA_OK:
        raise PAError("pa_decode_partitions", st)


def pa_merge(plan, context_lens, out, lse, workspace, stream=None) -> None:
    et = _TORCH_DTYPE.get(plan.dtype, torch.float16)
    st = load().pa_merge(ctypes.byref(plan), _dev_ptr(context_lens, "context_lens", torch.int32),
                         _dev_ptr(out, "out", et), _dev_ptr(lse, "lse", torch.float32),
                         _dev_ptr(workspace, "workspace"), _stream_ptr(stream))
    if st != PA_OK:
        raise PAError("pa_merge", st)


def pa_decode_static(plan, q, k_cache, v_cache, block_tables, context_lens, scale, window, out,
                     lse, stream=None) -> None:
    """pa_decode with the library's built-in scratch instead of a workspace,
    for callers that must not allocate device memory (see include/pa.h)."""
    args = _decode_args(plan, q, k_cache, v_cache, block_tables, context_lens, scale, window,
                        out, lse, None, stream)
    st = load().pa_decode_static(*args[:10], args[11])
    if st != PA_OK:
        raise PAError("pa_decode_static", st)


def pa_get_error(workspace, stream=None) -> int:
    """Synchronise and read the device error word (PA_DEVERR_* bits), leaving it set."""
    v = ctypes.c_int(0)
    st = load().pa_get_error(_dev_ptr(workspace, "workspace"), _stream_ptr(stream),
                             ctypes.byref(v))
    if st != PA_OK:
        raise PAError("pa_get_error", st)
    return int(v.value) & 0xFFFFFFFF


def pa_get_error_ex(workspace, stream=None, clear=True) -> int:
    """Synchronise, read the device error word and (clear=True) reset it to 0."""
    v = ctypes.c_uint(0)
    st = load().pa_get_error_ex(_dev_ptr(workspace, "workspace"), _stream_ptr(stream),
                                1 if clear else 0, ctypes.byref(v))
    if st != PA_OK:
        raise PAError("pa_get_error_ex", st)
    return int(v.value)


def new_workspace(plan, device=None) -> torch.Tensor:
    """Zero-filled device workspace of plan.workspace_bytes (uint8)."""
    return torch.zeros(max(int(plan.workspace_bytes), 256), dtype=torch.uint8, device=device)


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, window=0,
           partition_size=0, max_context_len=None, rope_theta=0.0, stream=None):
    """Convenience call: plan, allocate out/lse/workspace with torch, decode.

    The element type (fp16, bf16 or fp32) follows q; k_cache and v_cache must
    match it.  max_context_len defaults to the table's capacity
    (block_tables.shape[1] * page_size), which needs no device read.
    rope_theta > 0 applies the in-kernel rotary embedding with that base.
    Returns (out, lse, plan, device_error) -- device_error is read back, so
    this call synchronises.
    """
    dtypes = {v: k for k, v in _TORCH_DTYPE.items()}
    if q.dtype not in dtypes:
        raise TypeError(f"q must be fp16, bf16 or fp32, got {q.dtype}")
    B, Hq, D = q.shape
    num_pages, Hkv, ps, _ = k_cache.shape
    maxp = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = maxp * ps
    with torch.cuda.device(q.device):  # num_sms 0: plan for q's device, asking it
        plan = pa_plan_ex(B, Hq, Hkv, D, ps, num_pages, maxp, max_context_len, window,
                          partition_size, 0, dtype=dtypes[q.dtype], kernel=0,
                          rope_theta=rope_theta)
    out = torch.empty((B, Hq, D), dtype=q.dtype, device=q.device)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    ws = new_workspace(plan, q.device)
    pa_decode(plan, q, k_cache, v_cache, block_tables, context_lens, scale, window, out, lse, ws,
              stream)
    err = pa_get_error(ws, stream)
    return out, lse, plan, err
