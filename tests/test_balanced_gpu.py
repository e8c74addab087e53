"""Work-balanced partitions (pa_plan_t.balanced) against the fp64 oracle.

A balanced plan gives the X CTAs along grid.x of each (KV head, head chunk)
to the whole batch: the partition size is chosen on the device from the
actual lengths, so a long sequence gets more CTAs than a short one, and each
sequence's partials are merged by its last CTA.  These tests force such plans
(partition_size = PA_PARTITION_BALANCED) on the shapes where the mapping has
corners: ragged lengths with empty and single-token sequences, windows, one
long sequence among short ones (more partials than one load round of the
last-CTA merge takes), the largest batch the mapping spreads, bf16, bad page
ids and lengths, and a copy timeout; with either merge (the last CTA of each
group, or the merge kernel working out the same partition size)."""
import numpy as np
import pytest

import gpu_helpers
import oracle
import paged_kv_gqa_pa_gb300 as pa
from gpu_helpers import assert_matches_oracle, run_gpu
from paged_kv_gqa_pa_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

BAL = binding.PA_PARTITION_BALANCED


@pytest.fixture(autouse=True)
def tensor_core_kernel():
    gpu_helpers.KERNEL = "mma"
    yield
    gpu_helpers.KERNEL = None


def _check_plan(plan, B, fused=None):
    assert plan.balanced > B and plan.num_partitions == plan.balanced
    assert plan.cluster == 0 and plan.parts_per_cta == 1
    if fused is not None:
        assert plan.merge_in_kernel == fused


# Both merges: the last CTA of each group (fused 1), or the merge kernel,
# which works out the same partition size from the lengths (fused 0).
@pytest.mark.parametrize("fused", [1, 0])
def test_ragged_workload_full_size(fused):
    case = workloads.workload("batch8_ragged_d128")
    out, lse, err, plan = run_gpu(case, partition_size=BAL, guard=64, merge_in_kernel=fused)
    assert err == 0
    _check_plan(plan, case.B, fused)
    assert_matches_oracle(case, out, lse, what="balanced batch8_ragged_d128")


@pytest.mark.parametrize("fused", [1, 0])
@pytest.mark.parametrize("window", [0, 1000])
def test_ragged_with_empty_and_unit_sequences(window, fused):
    lens = [0, 1, 4096, 17, 0, 1000, 2, 3333]
    case = workloads.make_case("r", len(lens), 32, 8, 128, lens, seed=1400, window=window)
    out, lse, err, plan = run_gpu(case, partition_size=BAL, guard=64, merge_in_kernel=fused)
    assert err == 0
    _check_plan(plan, case.B, fused)
    assert np.all(out[[0, 4]] == 0) and np.all(np.isneginf(lse[[0, 4]]))
    assert_matches_oracle(case, out, lse, what=f"balanced ragged, window {window}")


@pytest.mark.parametrize("fused", [1, 0])
def test_one_long_sequence_many_partials(fused):
    # Nearly all of the grid goes to the long sequence: its partials exceed
    # one load round of the last-CTA merge (24 per thread at one thread per item).
    case = workloads.make_case("long1", 3, 32, 8, 128, [1, 60000, 5], seed=1401)
    out, lse, err, plan = run_gpu(case, partition_size=BAL, merge_in_kernel=fused)
    assert err == 0
    _check_plan(plan, case.B, fused)
    pages = -(-60000 // 16)
    pp = -(-(pages + 2) // (plan.balanced - 3))
    assert -(-pages // pp) > 24
    assert_matches_oracle(case, out, lse, what="balanced, one long sequence")


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 8, 8), (96, 12, 4), (256, 8, 4)])
def test_head_dims_and_groups(D, Hq, Hkv):
    lens = [3000, 5, 700, 1, 2222, 16, 17, 0, 64]
    case = workloads.make_case("dims", len(lens), Hq, Hkv, D, lens, seed=1402 + D)
    out, lse, err, plan = run_gpu(case, partition_size=BAL)
    assert err == 0
    _check_plan(plan, case.B)
    assert_matches_oracle(case, out, lse, what=f"balanced D{D}")


@pytest.mark.parametrize("fused", [1, 0])
def test_largest_batch(fused):
    rng = np.random.default_rng(1403)
    lens = rng.integers(0, 600, size=128).tolist()
    case = workloads.make_case("b128", 128, 8, 2, 64, lens, seed=1404)
    out, lse, err, plan = run_gpu(case, partition_size=BAL, merge_in_kernel=fused)
    assert err == 0
    _check_plan(plan, case.B)
    assert_matches_oracle(case, out, lse, what="balanced, 128 sequences")


def test_bf16_window():
    lens = [8192, 100, 5000, 4097]
    case = workloads.make_case("bfw", 4, 8, 4, 256, lens, seed=1405, window=4096, q_std=3.0,
                               dtype="bf16")
    out, lse, err, plan = run_gpu(case, partition_size=BAL)
    assert err == 0
    _check_plan(plan, case.B)
    assert_matches_oracle(case, out, lse, what="balanced bf16 window")


@pytest.mark.parametrize("fused", [1, 0])
def test_bad_page_and_bad_length_only_poison_their_sequence(fused):
    lens = [700, 1200, 90, 2000]
    case = workloads.make_case("badb", 4, 8, 2, 128, lens, seed=1406)
    ref_out, ref_lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                                     case.context_lens, case.scale, case.window)
    orig = int(case.block_tables[1, 5])
    case.block_tables[1, 5] = case.num_pages
    out, lse, err, plan = run_gpu(case, partition_size=BAL, max_context_len=2000,
                                  merge_in_kernel=fused)
    _check_plan(plan, case.B)
    assert err & binding.PA_DEVERR_BAD_PAGE
    assert np.isnan(out[1]).all() and np.isnan(lse[1]).all()
    good = [0, 2, 3]
    assert np.abs(lse[good] - ref_lse[good]).max() <= gpu_helpers.LSE_TOL
    assert gpu_helpers.rel_l2(out[good], ref_out[good]) <= gpu_helpers.REL_L2_TOL
    # A length beyond the plan's bound: that sequence is NaN, the rest exact.
    case.block_tables[1, 5] = orig
    out, lse, err, plan = run_gpu(case, partition_size=BAL, max_context_len=1500,
                                  merge_in_kernel=fused)
    assert err & binding.PA_DEVERR_BAD_LENGTH
    assert np.isnan(out[3]).all() and np.isnan(lse[3]).all()
    good = [0, 1, 2]
    assert np.abs(lse[good] - ref_lse[good]).max() <= gpu_helpers.LSE_TOL
    assert gpu_helpers.rel_l2(out[good], ref_out[good]) <= gpu_helpers.REL_L2_TOL


def test_copy_timeout_then_clean_call():
    case = workloads.make_case("stallb", 3, 8, 2, 128, [300, 40, 2000], seed=1407)
    out, lse, err, plan = run_gpu(case, partition_size=BAL, test_stall_bytes=16)
    assert err & binding.PA_DEVERR_TIMEOUT
    assert np.isnan(out).all() and np.isnan(lse).all()
    out, lse, err, plan = run_gpu(case, partition_size=BAL)
    assert err == 0
    assert_matches_oracle(case, out, lse, what="balanced after a timeout")


def test_agrees_with_fixed_partitions():
    case = workloads.workload("gemma2-2b_ctx8192_win4096")
    a = run_gpu(case, partition_size=BAL)
    b = run_gpu(case)
    assert a[2] == 0 and b[2] == 0
    assert gpu_helpers.rel_l2(a[0], b[0]) <= gpu_helpers.REL_L2_TOL
    assert np.abs(a[1] - b[1]).max() <= gpu_helpers.LSE_TOL
    assert_matches_oracle(case, a[0], a[1], what="balanced gemma2")


@pytest.mark.parametrize("lens,Hq,Hkv,D", [
    ([5000], 32, 8, 128),                 # one sequence: X CTAs on it alone
    ([2000, 700, 3100], 64, 4, 64),       # g = 16: two head chunks of 8 per KV head
    ([0, 0, 0, 4500], 4, 2, 256),         # only the last sequence attends anything
])
def test_edge_shapes(lens, Hq, Hkv, D):
    case = workloads.make_case("edge", len(lens), Hq, Hkv, D, lens, seed=1410 + len(lens))
    out, lse, err, plan = run_gpu(case, partition_size=BAL, guard=32)
    assert err == 0
    _check_plan(plan, case.B)
    assert plan.heads_per_cta * (Hq // Hkv // plan.heads_per_cta) == Hq // Hkv
    empty = [i for i, L in enumerate(lens) if L == 0]
    if empty:
        assert np.all(out[empty] == 0) and np.all(np.isneginf(lse[empty]))
    assert_matches_oracle(case, out, lse, what=f"balanced edge {lens}")


@pytest.mark.parametrize("fused", [1, 0])
@pytest.mark.parametrize("Hq,Hkv,D", [(64, 8, 128), (24, 4, 256)])
def test_wide_groups(Hq, Hkv, D, fused):
    """8 heads at D 128 (256 head-column items) and 6 at D 256 (384): the
    last CTA of a group merges its items kThreads at a time (fused 1); the
    planner gives these shapes the merge kernel (fused 0)."""
    lens = [9000, 120, 40, 2600]
    case = workloads.make_case("wide", len(lens), Hq, Hkv, D, lens, seed=1420 + D)
    out, lse, err, plan = run_gpu(case, partition_size=BAL, merge_in_kernel=fused)
    assert err == 0
    _check_plan(plan, case.B, fused)
    assert plan.heads_per_cta * (D // 4) > 128
    assert_matches_oracle(case, out, lse, what=f"balanced wide group Hq{Hq} D{D}")
