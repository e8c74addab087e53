"""GPU parity of the cluster merge: the partitions of each (sequence, KV head,
head chunk) run as one thread-block cluster and merge through distributed
shared memory inside the partition kernel (tensor-core kernel, plan.cluster).

Every case runs once with the cluster merge forced and once with it forbidden
(the merge kernel or the last-CTA merge), and both are compared with the fp64
oracle at the parity bar of tests/gpu_helpers.py."""
import numpy as np
import pytest

import oracle
import paged_kv_gqa_pa_gb300 as pa
from gpu_helpers import assert_matches_oracle, run_gpu
from paged_kv_gqa_pa_gb300 import workloads
import gpu_helpers

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tensor_core_kernel():
    gpu_helpers.KERNEL = "mma"
    yield
    gpu_helpers.KERNEL = None


def _both(case, **kw):
    """(out, lse, err, plan) with the cluster merge, then without it."""
    return run_gpu(case, cluster=True, **kw), run_gpu(case, cluster=False, **kw)


# Cluster sizes 2, 3, 7, 8 (portable) and 9, 16 (non-portable) over head dims
# and element types; the lengths include 1, page edges and ragged tails.
@pytest.mark.parametrize("D,Hq,Hkv,dtype", [(64, 4, 1, "f16"), (96, 8, 2, "f16"),
                                            (128, 32, 8, "f16"), (256, 24, 4, "f16"),
                                            (128, 8, 2, "bf16")])
@pytest.mark.parametrize("lens,S", [([1, 17, 40, 100], 32), ([255, 256, 257, 512], 96),
                                    ([3060, 2999], 208), ([4096, 4000], 256),
                                    ([1500, 1501], 176), ([1537, 33], 96)])
def test_cluster_merge_matches_oracle(D, Hq, Hkv, dtype, lens, S):
    case = workloads.make_case("cl", len(lens), Hq, Hkv, D, lens, seed=1100 + D, dtype=dtype,
                               partition_size=S, q_std=2.0)
    P = -(-max(lens) // S)
    if not 2 <= P <= 16:
        pytest.skip(f"{P} partitions: no cluster")
    (o1, l1, e1, p1), (o2, l2, e2, p2) = _both(case, guard=32)
    assert e1 == 0 and e2 == 0
    assert p1.cluster == P and p2.cluster == 0
    ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                        case.context_lens, case.scale, case.window, dtype=case.dtype)
    assert_matches_oracle(case, o1, l1, ref=ref, what=f"cluster D{D} {dtype} P{P}")
    assert_matches_oracle(case, o2, l2, ref=ref, what=f"no cluster D{D} {dtype} P{P}")


@pytest.mark.parametrize("Hq,Hkv,D,lens,S", [
    (16, 2, 256, [700, 1024, 513], 512),   # 8 heads x 64 columns over 2 CTAs: 256 items each
    (24, 4, 256, [900, 1000], 512),        # 6 heads: 192 items each
    (32, 4, 128, [300, 2000], 1024),       # 8 heads at D 128: 128 items each
])
def test_cluster_of_two_merges_two_rounds_per_thread(Hq, Hkv, D, lens, S):
    """The smallest cluster gives each CTA the most (head, column) items to
    merge: more than one per thread at D = 256, held in registers across the
    second cluster barrier and stored after it."""
    case = workloads.make_case("cl2", len(lens), Hq, Hkv, D, lens, seed=1230 + D, q_std=2.0,
                               partition_size=S)
    out, lse, err, plan = run_gpu(case, cluster=True)
    assert err == 0 and plan.cluster == 2
    assert_matches_oracle(case, out, lse, what=f"cluster of 2, {Hq}/{Hkv} heads, D {D}")


def test_cluster_ragged_batch_with_empty_sequences():
    # Sequences shorter than the cluster's span leave CTAs with nothing to
    # attend; empty sequences give out = 0, lse = -inf.
    lens = [0, 1, 4096, 17, 0, 1000, 2, 3333]
    case = workloads.make_case("clr", len(lens), 32, 8, 128, lens, seed=1200,
                               partition_size=512)
    (out, lse, err, plan), _ = _both(case, guard=64)
    assert err == 0 and plan.cluster == 8
    assert np.all(out[[0, 4]] == 0) and np.all(np.isneginf(lse[[0, 4]]))
    assert_matches_oracle(case, out, lse, what="cluster ragged")


def test_cluster_all_empty_batch():
    case = workloads.make_case("cle", 2, 8, 2, 128, [0, 0], seed=1201, partition_size=16,
                               pool_pages=8, max_pages_per_seq=4)
    out, lse, err, plan = run_gpu(case, max_context_len=64, cluster=True)
    assert err == 0 and plan.cluster == 4
    assert np.all(out == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("window", [1, 100, 1000, 4096])
def test_cluster_sliding_window(window):
    case = workloads.make_case("clw", 3, 8, 4, 256, [8192, 5000, 700], seed=1202, window=window,
                               q_std=3.0)
    for S in (64, 512):
        case.partition_size = S
        span = (window - 1 + 15) // 16 + 1
        if not 2 <= -(-span // (S // 16)) <= 16:
            continue
        out, lse, err, _ = run_gpu(case, cluster=True)
        assert err == 0
        assert_matches_oracle(case, out, lse, what=f"cluster W{window} S{S}")


def test_cluster_single_token_is_v_row_bit_exact():
    case = workloads.make_case("cl1", 4, 16, 2, 256, [1, 1, 1, 1], seed=1203, q_std=3.0,
                               max_pages_per_seq=4)
    out, lse, err, plan = run_gpu(case, max_context_len=64, partition_size=16, cluster=True)
    assert err == 0 and plan.cluster == 4
    for b in range(4):
        page = case.block_tables[b, 0]
        for h in range(16):
            assert np.array_equal(out[b, h], case.v_cache[page, h // 8, 0].astype(np.float64))


@pytest.mark.parametrize("bad", ["past_pool", "minus_one"])
def test_cluster_bad_page_sets_error_and_nan_rows(bad):
    case = workloads.make_case("clb", 3, 8, 2, 128, [700, 1200, 90], seed=1204,
                               partition_size=128)
    ref_out, ref_lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                                     case.context_lens, case.scale)
    case.block_tables[1, 5] = case.num_pages if bad == "past_pool" else -1
    out, lse, err, plan = run_gpu(case, guard=64, cluster=True)
    assert plan.cluster == 10
    assert err & pa.binding.PA_DEVERR_BAD_PAGE
    assert np.isnan(out[1]).all() and np.isnan(lse[1]).all()
    sub = workloads.Case(**{**case.__dict__, "q": case.q[[0, 2]],
                            "block_tables": case.block_tables[[0, 2]],
                            "context_lens": case.context_lens[[0, 2]]})
    assert_matches_oracle(sub, out[[0, 2]], lse[[0, 2]], ref=(ref_out[[0, 2]], ref_lse[[0, 2]]),
                          what="cluster good rows")


def test_cluster_context_longer_than_plan_bound():
    case = workloads.make_case("cll", 2, 4, 1, 64, [300, 1000], seed=1205, partition_size=64)
    ref_out, ref_lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                                     case.context_lens, case.scale)
    out, lse, err, plan = run_gpu(case, max_context_len=512, cluster=True)
    assert plan.cluster == 8
    assert err & pa.binding.PA_DEVERR_BAD_LENGTH
    assert np.isnan(out[1]).all() and np.isnan(lse[1]).all()
    assert np.abs(lse[0] - ref_lse[0]).max() <= 1e-4


def test_cluster_plan_validation():
    case = workloads.make_case("clv", 1, 8, 2, 128, [1000], seed=1206, partition_size=128)
    plan = pa.pa_plan_ex(1, 8, 2, 128, 16, case.num_pages, case.max_pages_per_seq, 1000, 0, 128,
                         152, kernel=pa.binding.PA_KERNEL_MMA)
    dev = gpu_helpers.to_device(case)
    import torch
    out = torch.empty((1, 8, 128), dtype=torch.float16, device="cuda")
    lse = torch.empty((1, 8), dtype=torch.float32, device="cuda")
    ws = pa.new_workspace(plan, "cuda")
    for field, value in (("cluster", 17), ("cluster", 5), ("cluster", -1)):
        bad = pa.binding.pa_plan_t.from_buffer_copy(plan)
        setattr(bad, field, value)
        with pytest.raises(pa.binding.PAError):
            pa.pa_decode(bad, dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"], case.scale, 0,
                         out, lse, ws)
    bad = pa.binding.pa_plan_t.from_buffer_copy(plan)
    bad.cluster = bad.num_partitions
    bad.parts_per_cta = 2
    with pytest.raises(pa.binding.PAError):
        pa.pa_decode(bad, dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"], case.scale, 0, out,
                     lse, ws)


@pytest.mark.parametrize("D,dtype,rope", [(256, 0, 0.0), (128, 0, 0.0), (64, 1, 0.0),
                                          (96, 0, 0.0), (128, 0, 10000.0), (256, 1, 10000.0)])
def test_plan_for_this_device_asks_it_and_agrees_with_the_gb300_table(D, dtype, rope):
    """A plan for the current device (num_sms = 0) takes the clusters a wave
    holds from cudaOccupancyMaxActiveClusters; a plan for an explicit SM count
    takes them from the table measured on a 152-SM GB300.  On that part the
    two must pick the same cluster for every group count: the sweep crosses
    every cluster size's threshold."""
    import torch
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the table was measured on the 152-SM GB300")
    for B in range(1, 161):
        args = (B, 4, 1, D, 16, 100000, 128, 2048, 0, 0)
        asked = pa.pa_plan_ex(*args, 0, dtype=dtype, rope_theta=rope)
        table = pa.pa_plan_ex(*args, 152, dtype=dtype, rope_theta=rope)
        assert asked.num_sms == 152
        assert (asked.cluster, asked.num_partitions, asked.partition_size) == \
            (table.cluster, table.num_partitions, table.partition_size), (B, D, dtype, rope)


@pytest.mark.parametrize("D,dtype", [(128, "f16"), (96, "f16"), (128, "bf16"), (96, "bf16"),
                                     (256, "f16"), (256, "bf16")])
@pytest.mark.parametrize("lens,window", [([16384], 0), ([8000], 0), ([12345], 4096), ([1], 0)])
def test_deep_ring_cluster_instance_matches_the_default_one(D, dtype, lens, window):
    """The deep-ring cluster instance (2 CTAs per SM, more pages in flight per
    warp) walks the same pages in the same order as the default one: results
    are bitwise equal, and match the oracle."""
    case = workloads.make_case("deep", len(lens), 32, 8, D, lens, seed=1240 + D, window=window,
                               dtype=dtype, q_std=2.0)
    a = run_gpu(case, guard=32, deep_ring=1)
    b = run_gpu(case, guard=32, deep_ring=0)
    assert a[2] == 0 and b[2] == 0
    if lens[0] > 1:
        assert a[3].cluster > 1 and a[3].deep_ring == 1
    assert np.array_equal(a[0], b[0], equal_nan=True) and np.array_equal(a[1], b[1], equal_nan=True)
    assert_matches_oracle(case, a[0], a[1], what=f"deep ring D{D} {dtype} {lens}")
