"""GPU test of the tensor-core kernel's pre-wait prefetch hints.

Before its programmatic-dependent-launch wait the partition kernel reads the
sequence length and each warp's first page ids as hints and requests those
pages into L2; after the wait it reads everything again.  Here a helper kernel
on the same stream lets the decode start early, waits, and only then writes
the real block table and lengths: the old table points at the pool's
NaN-filled slack pages, so a stale hint that reached the output would poison
it.  The result must match the fp64 oracle on the new values."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_pa_gb300 as pa
from gpu_helpers import assert_matches_oracle, ensure_built, to_device
from paged_kv_gqa_pa_gb300 import workloads

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def writer():
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libpdl_writer.so")
    src = os.path.join(HERE, "cuda", "pdl_writer.cu")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                        "-Xcompiler", "-fPIC", src, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.launch_delayed_copy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_ulonglong, ctypes.c_void_p]
    return lib


def _slack_pages(case):
    used = set(int(x) for x in case.block_tables.ravel() if x >= 0)
    return np.array(sorted(set(range(case.num_pages)) - used), dtype=np.int32)


# lens_delta: how far the old lengths (the hints) lie from the real ones.  The
# kernel stages the block-table entries of the hint's range plus a page on
# either side together with the real length: with a window, 5 tokens keep the
# real range inside them (the entries are reused, shifted), 37 tokens move it
# out (they are loaded again).
@pytest.mark.parametrize("window", [0, 1000])
@pytest.mark.parametrize("lens_delta", [0, 5, 37])
@pytest.mark.parametrize("plan_kind", ["cluster", "merge_kernel", "unsplit"])
def test_stale_hints_are_replaced(writer, lens_delta, plan_kind, window):
    ensure_built()
    lens = [3000, 1200, 2049, 77]
    case = workloads.make_case("pdl", len(lens), 16, 4, 128, lens, seed=1500, q_std=2.0,
                               window=window)
    slack = _slack_pages(case)
    assert len(slack) > 0
    # The old values: every table entry a NaN slack page, lengths near the cap.
    old_bt = slack[np.arange(case.block_tables.size) % len(slack)].reshape(case.block_tables.shape)
    old_cl = case.context_lens.copy()
    if lens_delta:
        old_cl = np.minimum(old_cl + lens_delta, case.max_context_len).astype(np.int32)
    dev = to_device(case)
    new_bt, new_cl = dev["bt"].clone(), dev["cl"].clone()
    dev["bt"].copy_(torch.from_numpy(old_bt))
    dev["cl"].copy_(torch.from_numpy(old_cl))
    B, Hq, D = case.q.shape
    S = {"cluster": 256, "merge_kernel": 96, "unsplit": 4096}[plan_kind]
    plan = pa.pa_plan(B, Hq, case.Hkv, D, 16, case.num_pages, case.max_pages_per_seq,
                      case.max_context_len, window, S,
                      torch.cuda.get_device_properties(0).multi_processor_count)
    if plan_kind == "cluster":
        plan.cluster, plan.parts_per_cta, plan.merge_in_kernel = plan.num_partitions, 1, 0
        assert 2 <= plan.num_partitions <= 16
    elif plan_kind == "merge_kernel":
        plan.cluster, plan.merge_in_kernel = 0, 0
    assert plan.kernel == 2 and plan.prewait_prefetch > 0
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = pa.new_workspace(plan, "cuda")
    stream = torch.cuda.current_stream()
    assert writer.launch_delayed_copy(new_bt.data_ptr(), dev["bt"].data_ptr(), new_bt.numel(),
                                      new_cl.data_ptr(), dev["cl"].data_ptr(), new_cl.numel(),
                                      20000, stream.cuda_stream) == 0
    pa.pa_decode(plan, dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"], case.scale, window,
                 out, lse, ws, stream)
    assert pa.pa_get_error(ws) == 0
    torch.cuda.synchronize()
    assert torch.equal(dev["bt"], new_bt) and torch.equal(dev["cl"], new_cl)
    assert_matches_oracle(case, out.double().cpu().numpy(), lse.double().cpu().numpy(),
                          what=f"stale hints {plan_kind} lens_delta={lens_delta} window={window}")
