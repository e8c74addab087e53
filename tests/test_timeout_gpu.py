"""The tensor-core kernel's copy-timeout path, exercised without any fault.

Every wait of the kernel on a page copy is bounded: after 1 s it sets
PA_DEVERR_TIMEOUT in the device error word, gives its own copies in flight a
bounded time to land, writes NaN rows and returns, and the context stays
usable.  The plan's test hook test_stall_bytes makes each warp's first copy
expect more bytes than it carries, so its barrier never completes and the
bounded wait runs out -- a wait that nothing completes, not a fault.  Each
case checks the status and the NaN rows, then a normal call on the same
workspace and context, which must match the fp64 oracle."""
import numpy as np
import pytest

import gpu_helpers
import paged_kv_gqa_pa_gb300 as pa
from gpu_helpers import assert_matches_oracle, run_gpu
from paged_kv_gqa_pa_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tensor_core_kernel():
    gpu_helpers.KERNEL = "mma"
    yield
    gpu_helpers.KERNEL = None


PLANS = {
    "unsplit": dict(partition_size=4096),
    "merge_kernel": dict(partition_size=64, cluster=False, merge_in_kernel=0),
    "last_cta_merge": dict(partition_size=128, merge_in_kernel=1),
    "cluster": dict(partition_size=128, cluster=True),
    "one_warp_per_partition": dict(partition_size=32, parts_per_cta=4, merge_in_kernel=0),
}


@pytest.mark.parametrize("plan_kind", sorted(PLANS))
def test_copy_timeout_reports_nan_and_the_next_call_is_clean(plan_kind):
    case = workloads.make_case("stall", 2, 8, 2, 128, [300, 40], seed=1700)
    kw = PLANS[plan_kind]
    out, lse, err, plan = run_gpu(case, test_stall_bytes=16, **kw)
    assert plan.test_stall_bytes == 16
    assert err & binding.PA_DEVERR_TIMEOUT
    assert np.isnan(out).all() and np.isnan(lse).all()
    out, lse, err, plan = run_gpu(case, **kw)
    assert err == 0 and plan.test_stall_bytes == 0
    assert_matches_oracle(case, out, lse, what=f"after a timeout, {plan_kind}")
