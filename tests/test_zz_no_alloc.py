"""pa_decode_static: the decode entry point that allocates nothing.

It exists for callers that cannot hand the library a workspace: engines and
plugins that are given only their own input and output buffers, and loops that
must never enter the allocator (cudaMalloc can synchronise the device).  The partition
partials then go to a scratch array built into the library.  These tests call
it through the C ABI (ctypes on libpa_gb300.so) and check it against pa_decode
with a caller workspace, on two calls in a row with different problems (the
second call finds the first call's partials still in the shared scratch).

The file is named to be collected last, so that a stop-at-first-failure run
has already run every other test when it gets here."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_gqa_pa_gb300 as pa
from gpu_helpers import LSE_TOL, REL_L2_TOL, ensure_built, rel_l2, to_device
from paged_kv_gqa_pa_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

STATIC_BYTES = 32 << 20  # PA_STATIC_WORKSPACE_BYTES in include/pa.h


def _plan(case, S):
    B, Hq, D = case.q.shape
    return pa.pa_plan(B, Hq, case.Hkv, D, 16, case.num_pages, case.max_pages_per_seq,
                      case.max_context_len, case.window, S,
                      torch.cuda.get_device_properties(0).multi_processor_count)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _run(case, plan, static):
    dev = to_device(case)
    B, Hq, D = case.q.shape
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    lib = pa.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if static:
        st = lib.pa_decode_static(ctypes.byref(plan), _ptr(dev["q"]), _ptr(dev["k"]),
                                  _ptr(dev["v"]), _ptr(dev["bt"]), _ptr(dev["cl"]),
                                  ctypes.c_float(case.scale), case.window, _ptr(out), _ptr(lse),
                                  stream)
    else:
        ws = pa.new_workspace(plan, "cuda")
        st = lib.pa_decode(ctypes.byref(plan), _ptr(dev["q"]), _ptr(dev["k"]), _ptr(dev["v"]),
                           _ptr(dev["bt"]), _ptr(dev["cl"]), ctypes.c_float(case.scale),
                           case.window, _ptr(out), _ptr(lse), _ptr(ws), stream)
    assert st == binding.PA_OK, pa.pa_status_string(st)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def _close(a, b):
    (oa, la), (ob, lb) = a, b
    assert not np.isnan(oa).any()
    assert rel_l2(oa, ob) <= REL_L2_TOL
    fin = np.isfinite(lb)
    assert np.array_equal(np.isfinite(la), fin)
    if fin.any():
        assert np.abs(la[fin] - lb[fin]).max() <= LSE_TOL


@pytest.mark.parametrize("kernel", [binding.PA_KERNEL_MMA, binding.PA_KERNEL_SIMT])
def test_static_scratch_matches_workspace_path_two_calls(kernel):
    ensure_built()
    first = workloads.make_case("s1", 3, 16, 2, 128, [3000, 17, 1500], seed=901, window=0)
    second = workloads.make_case("s2", 2, 24, 4, 256, [20000, 777], seed=902, window=5000,
                                 q_std=2.0)
    for case, S in ((first, 256), (second, 512)):
        plan = _plan(case, S)
        plan.kernel = kernel
        assert plan.num_partitions > 1 and 0 < plan.workspace_bytes <= STATIC_BYTES
        ref = _run(case, plan, static=False)
        got = _run(case, plan, static=True)
        _close(got, ref)


def test_static_scratch_rejects_oversized_plan():
    ensure_built()
    # 4 sequences x 64 query heads x 4096 partitions of 16 tokens need far more
    # than the built-in scratch for their partials.
    plan = pa.pa_plan(4, 64, 8, 256, 16, 1 << 16, 4096, 65536, 0, 16, 152)
    assert plan.workspace_bytes > STATIC_BYTES
    lib = pa.load()
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: rejected before any launch
    st = lib.pa_decode_static(ctypes.byref(plan), fake, fake, fake, fake, fake,
                              ctypes.c_float(0.1), 0, fake, fake, None)
    assert st == binding.PA_ERR_WORKSPACE
