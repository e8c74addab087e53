"""GB300-native paged-KV grouped-query decode attention.

The C ABI (include/pa.h) lives in libpa_gb300.so, built from csrc/ for sm_103a;
``binding`` exposes it to Python under the same names.  The library is loaded
on the first call, never at import, so ``workloads`` (the seeded input
generator) imports without a GPU.
"""
from .binding import (PAError, decode, load, new_workspace, pa_decode, pa_decode_partitions,
                      pa_decode_static, pa_get_error, pa_get_error_ex, pa_merge, pa_plan,
                      pa_plan_ex, pa_plan_t, pa_status_string, pa_version, prepare_decode)

__all__ = ["PAError", "decode", "load", "new_workspace", "pa_decode", "pa_decode_partitions",
           "pa_decode_static", "pa_get_error", "pa_get_error_ex", "pa_merge", "pa_plan",
           "pa_plan_ex", "pa_plan_t", "pa_status_string", "pa_version", "prepare_decode"]
