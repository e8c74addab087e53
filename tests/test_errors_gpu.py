"""Data-dependent faults on the GPU: a bad block-table entry or a context
length beyond the plan's bound is never read through.  The kernel sets a bit of
the device error word and writes NaN rows for the affected sequence; the other
sequences are unaffected.  Nothing here faults, traps or hangs the GPU: the bad
values are rejected by the kernel's own bounds checks before any access."""
import numpy as np
import pytest

import gpu_helpers
import oracle
import paged_kv_gqa_pa_gb300 as pa
from gpu_helpers import assert_matches_oracle, run_gpu
from paged_kv_gqa_pa_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["mma", "simt"], autouse=True)
def kernel_variant(request):
    """Run every test on both partition kernels (tensor-core and CUDA-core)."""
    gpu_helpers.KERNEL = request.param
    yield request.param
    gpu_helpers.KERNEL = None


def _ref_rows(case, rows):
    ref_out, ref_lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                                     case.context_lens, case.scale, case.window, dtype=case.dtype)
    return ref_out[rows], ref_lse[rows]


@pytest.mark.parametrize("fused", [0, 1])
@pytest.mark.parametrize("S", [0, 64, 4096])
@pytest.mark.parametrize("bad", ["past_pool", "minus_one"])
def test_bad_page_id_sets_error_and_nan_rows(S, bad, fused):
    if fused:  # partition sizes whose partition count the in-kernel merge takes (<= 8)
        S = {0: 512, 64: 256}.get(S, S)
    case = workloads.make_case("bad", 3, 8, 2, 128, [700, 1200, 90], seed=600, partition_size=S)
    good_ref = _ref_rows(case, [0, 2])
    case.block_tables[1, 5] = case.num_pages if bad == "past_pool" else -1
    out, lse, err, _ = run_gpu(case, guard=64, parts_per_cta=4 if S == 64 else None,
                               merge_in_kernel=fused)
    assert err & pa.binding.PA_DEVERR_BAD_PAGE
    assert np.isnan(out[1]).all() and np.isnan(lse[1]).all()
    sub = workloads.Case(**{**case.__dict__, "q": case.q[[0, 2]],
                            "block_tables": case.block_tables[[0, 2]],
                            "context_lens": case.context_lens[[0, 2]]})
    assert_matches_oracle(sub, out[[0, 2]], lse[[0, 2]], ref=good_ref, what="good rows")


@pytest.mark.parametrize("fused", [0, 1])
@pytest.mark.parametrize("S", [0, 64, 4096])
def test_context_longer_than_plan_bound(S, fused):
    case = workloads.make_case("long", 2, 4, 1, 64, [300, 1000], seed=601, partition_size=S)
    good_ref = _ref_rows(case, [0])
    # Plan for at most 512 tokens: sequence 1 (1000 tokens) breaks the bound.
    out, lse, err, _ = run_gpu(case, max_context_len=512, merge_in_kernel=fused)
    assert err & pa.binding.PA_DEVERR_BAD_LENGTH
    assert np.isnan(out[1]).all() and np.isnan(lse[1]).all()
    assert np.abs(lse[0] - good_ref[1][0]).max() <= 1e-4
    # The error word is cleared by the read: a clean call reports 0.
    out, lse, err, _ = run_gpu(case)
    assert err == 0


def test_negative_context_length():
    case = workloads.make_case("neg", 2, 4, 1, 64, [300, 100], seed=602)
    case.context_lens[1] = -5
    out, lse, err, _ = run_gpu(case, max_context_len=300)
    assert err & pa.binding.PA_DEVERR_BAD_LENGTH
    assert np.isnan(out[1]).all()
    assert not np.isnan(out[0]).any()


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f16", 96)])
def test_bad_page_on_wider_paths(dtype, D):
    if gpu_helpers.KERNEL == "simt" and D == 96:
        pytest.skip("the CUDA-core kernel is built for head dims 64/128/256")
    case = workloads.make_case("badw", 3, 8, 2, D, [700, 1200, 90], seed=610, partition_size=256,
                               dtype=dtype)
    good_ref = _ref_rows(case, [0, 2])
    case.block_tables[1, 7] = -1
    out, lse, err, _ = run_gpu(case, guard=64)
    assert err & pa.binding.PA_DEVERR_BAD_PAGE
    assert np.isnan(out[1]).all() and np.isnan(lse[1]).all()
    sub = workloads.Case(**{**case.__dict__, "q": case.q[[0, 2]],
                            "block_tables": case.block_tables[[0, 2]],
                            "context_lens": case.context_lens[[0, 2]]})
    assert_matches_oracle(sub, out[[0, 2]], lse[[0, 2]], ref=good_ref, what="good rows")
