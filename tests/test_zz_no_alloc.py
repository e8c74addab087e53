"""pa_decode_static: the decode entry point that allocates nothing.

It exists for callers that cannot hand the library a workspace: engines and
plugins that are given only their own input and output buffers, and loops that
must never enter the allocator (cudaMalloc can synchronise the device).  The
partition partials then go to a scratch array built into the library, shared
by every call on the device.

These tests call it through the C ABI (ctypes on libpa_gb300.so, and once
through the Python wrapper) and check it against pa_decode with a caller
workspace on the same plan -- the same kernels on the same inputs, so the
results must be bitwise equal -- and against the fp64 oracle.  Calls follow
each other with different plans, so each finds the previous call's contents
still in the shared scratch: partials of another layout, a device error word
left set by a timed-out call.  Every merge kind is covered (merge kernel,
last-CTA merge with its arrival counters, a work-balanced plan, cluster
merge).

The file is named to be collected last, so that a stop-at-first-failure run
has already run every other test when it gets here."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_gqa_pa_gb300 as pa
from gpu_helpers import assert_matches_oracle, ensure_built, to_device
from paged_kv_gqa_pa_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

STATIC_BYTES = 32 << 20  # PA_STATIC_WORKSPACE_BYTES in include/pa.h


def _plan(case, S, kernel=binding.PA_KERNEL_MMA, **fields):
    B, Hq, D = case.q.shape
    plan = pa.pa_plan_ex(B, Hq, case.Hkv, D, 16, case.num_pages, case.max_pages_per_seq,
                         case.max_context_len, case.window, S,
                         torch.cuda.get_device_properties(0).multi_processor_count,
                         kernel=kernel)
    for k, v in fields.items():
        setattr(plan, k, v)
    return plan


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _run(case, plan, static, via_binding=False):
    """One call; out and lse start as NaN so that a row nobody writes shows."""
    dev = to_device(case)
    B, Hq, D = case.q.shape
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    lib = pa.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if static and via_binding:
        pa.pa_decode_static(plan, dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"], case.scale,
                            case.window, out, lse)
    elif static:
        st = lib.pa_decode_static(ctypes.byref(plan), _ptr(dev["q"]), _ptr(dev["k"]),
                                  _ptr(dev["v"]), _ptr(dev["bt"]), _ptr(dev["cl"]),
                                  ctypes.c_float(case.scale), case.window, _ptr(out), _ptr(lse),
                                  stream)
        assert st == binding.PA_OK, pa.pa_status_string(st)
    else:
        ws = pa.new_workspace(plan, "cuda")
        st = lib.pa_decode(ctypes.byref(plan), _ptr(dev["q"]), _ptr(dev["k"]), _ptr(dev["v"]),
                           _ptr(dev["bt"]), _ptr(dev["cl"]), ctypes.c_float(case.scale),
                           case.window, _ptr(out), _ptr(lse), _ptr(ws), stream)
        assert st == binding.PA_OK, pa.pa_status_string(st)
        torch.cuda.synchronize()
        assert pa.pa_get_error(ws) == 0
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def _same(got, ref):
    """Bitwise equality of out (fp16 bits) and lse (fp32 bits)."""
    (og, lg), (orf, lrf) = got, ref
    assert torch.equal(og.view(torch.int16), orf.view(torch.int16)), "out differs"
    assert torch.equal(lg.view(torch.int32), lrf.view(torch.int32)), "lse differs"


def _check(case, plan, via_binding=False, what=""):
    """Static call vs workspace call (bitwise), then vs the oracle."""
    assert 0 < plan.workspace_bytes <= STATIC_BYTES
    ref = _run(case, plan, static=False)
    got = _run(case, plan, static=True, via_binding=via_binding)
    _same(got, ref)
    assert_matches_oracle(case, got[0].double().numpy(), got[1].double().numpy(), what=what)


@pytest.mark.parametrize("kernel", [binding.PA_KERNEL_MMA, binding.PA_KERNEL_SIMT])
def test_static_scratch_matches_workspace_path_two_calls(kernel):
    ensure_built()
    first = workloads.make_case("s1", 3, 16, 2, 128, [3000, 17, 1500], seed=901, window=0)
    second = workloads.make_case("s2", 2, 24, 4, 256, [20000, 777], seed=902, window=5000,
                                 q_std=2.0)
    for case, S in ((first, 256), (second, 512)):
        plan = _plan(case, S, kernel=kernel, cluster=0, merge_in_kernel=0)
        assert plan.num_partitions > 1
        _check(case, plan, what=f"static, kernel {kernel}, {case.name}")


def test_static_scratch_every_merge_kind_in_a_row():
    """Merge kernel, last-CTA merge (arrival counters in the shared array),
    work-balanced plan (partials of the whole batch spread over its CTAs) and
    cluster merge, one after another on the same scratch, the last one through
    the Python wrapper."""
    ensure_built()
    case = workloads.make_case("kinds", 2, 8, 2, 128, [1000, 700], seed=903, window=0)
    plans = {
        "merge_kernel": _plan(case, 64, cluster=0, merge_in_kernel=0),
        "last_cta_merge": _plan(case, 128, cluster=0, merge_in_kernel=1),
        "balanced": _plan(case, binding.PA_PARTITION_BALANCED),
        "cluster_merge": _plan(case, 128, merge_in_kernel=0, parts_per_cta=1),
    }
    assert plans["balanced"].balanced > 0
    plans["cluster_merge"].cluster = plans["cluster_merge"].num_partitions
    assert 2 <= plans["cluster_merge"].cluster <= 16
    assert plans["last_cta_merge"].num_partitions <= 8
    for kind, plan in plans.items():
        _check(case, plan, via_binding=(kind == "cluster_merge"), what=f"static, {kind}")


def test_static_counters_cleared_where_another_plan_left_partials():
    """A plan with few groups writes its partials right behind its small
    control region; the next plan has more (sequence, KV head) groups, so its
    arrival counters lie where those partials are.  The static call must clear
    them, or those groups' last-CTA merge never fires and their rows stay NaN."""
    ensure_built()
    a = workloads.make_case("few_groups", 1, 8, 2, 128, [4000], seed=904, window=0)
    plan_a = _plan(a, 64, cluster=0, merge_in_kernel=0)
    lens = [512, 300, 77, 480, 1, 512, 259, 400, 333]
    b = workloads.make_case("many_groups", 9, 16, 8, 64, lens, seed=905, window=0)
    plan_b = _plan(b, 64, cluster=0, merge_in_kernel=1)
    groups_b = 9 * 8
    assert plan_a.ctrl_bytes == 512 and plan_b.ctrl_bytes > 512 and groups_b > 64
    assert plan_a.num_partitions >= 8 and plan_b.merge_in_kernel == 1
    ref_b = _run(b, plan_b, static=False)
    _run(a, plan_a, static=True)   # leaves its partials at byte 512 on
    got_b = _run(b, plan_b, static=True)
    _same(got_b, ref_b)
    assert_matches_oracle(b, got_b[0].double().numpy(), got_b[1].double().numpy(),
                          what="static after another plan's partials")


@pytest.mark.parametrize("merge_in_kernel", [1, 0])
def test_static_call_after_a_timed_out_static_call_is_clean(merge_in_kernel):
    """The plan's test hook makes each warp's first copy wait for bytes that
    never come, so the bounded wait runs out (1 s) and the call returns NaN
    rows with the error word set in the shared array -- no fault.  The next
    static call must come out clean and bitwise equal to pa_decode."""
    ensure_built()
    case = workloads.make_case("stall_static", 2, 8, 2, 128, [900, 300], seed=906, window=0)
    plan = _plan(case, 128, cluster=0, merge_in_kernel=merge_in_kernel)
    stalled = binding.pa_plan_t.from_buffer_copy(plan)
    stalled.test_stall_bytes = 16
    out, lse = _run(case, stalled, static=True)
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
    _check(case, plan, what="static after a timed-out static call")


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
