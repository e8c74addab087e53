"""GPU parity of the tensor-core kernel's pre-wait L2 prefetch.

plan.prewait_prefetch requests each warp's first pages into L2 before the
programmatic-dependent-launch wait, from a sequence length and page ids read
as hints.  It may not change a result: every setting is compared with the fp64
oracle, over the plan shapes the kernel has (one partition, split with the
merge kernel, two partitions per CTA, the last-CTA merge, the cluster merge),
and a bad page id must still be reported and never prefetched from."""
import numpy as np
import pytest

import oracle
from gpu_helpers import assert_matches_oracle, run_gpu
from paged_kv_gqa_pa_gb300 import binding, workloads
import gpu_helpers

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tensor_core_kernel():
    gpu_helpers.KERNEL = "mma"
    yield
    gpu_helpers.KERNEL = None


PLANS = {
    "one_partition": dict(partition_size=4096),
    "merge_kernel": dict(partition_size=96, cluster=False, merge_in_kernel=0),
    "two_per_cta": dict(partition_size=64, parts_per_cta=2, merge_in_kernel=0),
    "last_cta_merge": dict(partition_size=1024, merge_in_kernel=1),
    "cluster": dict(partition_size=256, cluster=True),
}


@pytest.mark.parametrize("plan_kind", sorted(PLANS))
@pytest.mark.parametrize("pw", [1, 3, 8])
@pytest.mark.parametrize("D,Hq,Hkv,dtype", [(64, 8, 2, "f16"), (96, 8, 2, "f16"),
                                            (256, 24, 4, "f16"), (128, 16, 2, "bf16")])
def test_prefetch_settings_match_oracle(plan_kind, pw, D, Hq, Hkv, dtype):
    lens = [1, 700, 2049, 3333]
    case = workloads.make_case("pf", len(lens), Hq, Hkv, D, lens, seed=1300 + D + pw,
                               dtype=dtype, q_std=2.0, window=3000 if pw == 3 else 0)
    kw = dict(PLANS[plan_kind])
    out, lse, err, plan = run_gpu(case, guard=16, prewait_prefetch=pw, **kw)
    assert err == 0
    assert plan.prewait_prefetch == pw
    assert_matches_oracle(case, out, lse, what=f"{plan_kind} pw{pw} D{D} {dtype}")


def test_prefetch_skips_bad_page_ids():
    # A page id outside the pool in sequence 1 is reported and gives NaN rows
    # there; the prefetch hints never address it, and sequence 0 is unharmed.
    case = workloads.make_case("pfbad", 2, 8, 2, 128, [1000, 1000], seed=1390)
    case.block_tables[1, 5] = case.num_pages + 7
    for pw in (1, 8):
        out, lse, err, _ = run_gpu(case, partition_size=128, prewait_prefetch=pw)
        assert err & binding.PA_DEVERR_BAD_PAGE
        assert np.isnan(out[1]).all() and np.isnan(lse[1]).all()
        ref = oracle.decode(case.q[:1], case.k_cache, case.v_cache, case.block_tables[:1],
                            case.context_lens[:1], case.scale, case.window)
        assert gpu_helpers.rel_l2(out[:1], ref[0]) <= gpu_helpers.REL_L2_TOL


def test_prefetch_settings_are_checked():
    import paged_kv_gqa_pa_gb300 as pa
    import torch
    case = workloads.make_case("pfchk", 1, 8, 2, 128, [500], seed=1391)
    dev = gpu_helpers.to_device(case)
    plan = pa.pa_plan(1, 8, 2, 128, 16, case.num_pages, case.max_pages_per_seq, 500, 0, 128, 152)
    out = torch.empty((1, 8, 128), dtype=torch.float16, device="cuda")
    lse = torch.empty((1, 8), dtype=torch.float32, device="cuda")
    ws = pa.new_workspace(plan, "cuda")
    for field, value in (("prewait_prefetch", -1), ("prewait_prefetch", 9)):
        bad = binding.pa_plan_t.from_buffer_copy(plan)
        setattr(bad, field, value)
        with pytest.raises(pa.PAError) as e:
            pa.pa_decode(bad, dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"], case.scale, 0,
                         out, lse, ws)
        assert e.value.status == binding.PA_ERR_INVALID_ARG
