"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element
by element, on seeded inputs.

Bar: relative L2 <= 1e-3 over the fp16 output tensor and |dLSE| <= 1e-4
(tests/gpu_helpers.py); bit-exact where the result is exact (single-token
context, page placement, window >= context)."""
import math

import numpy as np
import pytest
import torch

import gpu_helpers
import oracle
from gpu_helpers import assert_matches_oracle, run_gpu, to_device
from paged_kv_gqa_pa_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["mma", "simt"], autouse=True)
def kernel_variant(request):
    """Run every test on both partition kernels (tensor-core and CUDA-core)."""
    gpu_helpers.KERNEL = request.param
    yield request.param
    gpu_helpers.KERNEL = None


# ---- the five measured workloads, at full size, in the plan the bench uses
@pytest.mark.parametrize("name", workloads.WORKLOAD_ORDER + workloads.EXTRA_ORDER)
def test_workload_full_size(name):
    case = workloads.workload(name)
    if gpu_helpers.KERNEL == "simt" and case.D == 96:
        pytest.skip("the CUDA-core kernel is built for head dims 64/128/256")
    if gpu_helpers.KERNEL == "mma" and case.dtype == "f32":
        pytest.skip("fp32 caches run on the CUDA-core kernel")
    out, lse, err, plan = run_gpu(case)
    assert err == 0
    rel = assert_matches_oracle(case, out, lse, what=name)
    if name.startswith("gqa6_ctx100k"):
        # 100000 tokens in 512-token partitions: 196 partitions, the last one
        # holding 160 tokens.
        assert plan.num_partitions == 196
    print(f"{name}: rel L2 {rel:.2e}, partitions {plan.num_partitions}")


# ---- context lengths of the pages' accuracy check (1 .. 3060, odd shard
# lengths), each head dim, forced split / no split / automatic
LENS = [1, 2, 15, 16, 17, 255, 256, 257, 511, 513, 3060]


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 4, 1), (128, 8, 2), (256, 6, 1)])
@pytest.mark.parametrize("partition_size", [0, 16, 64, 512, 4096])
def test_context_length_sweep(D, Hq, Hkv, partition_size):
    case = workloads.make_case("sweep", len(LENS), Hq, Hkv, D, LENS, seed=100 + D,
                               partition_size=partition_size)
    out, lse, err, plan = run_gpu(case)
    assert err == 0
    if partition_size == 4096:
        assert plan.num_partitions == 1  # whole context in one CTA, no merge
    assert_matches_oracle(case, out, lse, what=f"D{D} S{partition_size}")


@pytest.mark.parametrize("g", [1, 2, 3, 5, 7, 8, 12, 16])
def test_group_sizes(g):
    Hkv = 2
    case = workloads.make_case("g", 3, g * Hkv, Hkv, 128, [37, 700, 1500], seed=200 + g,
                               q_std=2.0)
    for S in (0, 128):
        case.partition_size = S
        out, lse, err, plan = run_gpu(case)
        assert err == 0
        assert_matches_oracle(case, out, lse, what=f"g{g} S{S}")


@pytest.mark.parametrize("window", [1, 7, 16, 100, 255, 1000, 3059, 3060, 5000])
def test_sliding_window(window):
    case = workloads.make_case("w", 3, 8, 4, 256, [3060, 1001, 40], seed=300, window=window,
                               q_std=3.0)
    for S in (0, 64, 2048):
        case.partition_size = S
        out, lse, err, _ = run_gpu(case)
        assert err == 0
        assert_matches_oracle(case, out, lse, what=f"W{window} S{S}")


def test_ragged_batch_with_empty_and_unit_sequences():
    lens = [0, 1, 4096, 17, 0, 1000, 2, 3333]
    case = workloads.make_case("r", len(lens), 32, 8, 128, lens, seed=400)
    for S in (0, 256, 4096):
        case.partition_size = S
        out, lse, err, _ = run_gpu(case, guard=64)
        assert err == 0
        assert np.all(out[[0, 4]] == 0) and np.all(np.isneginf(lse[[0, 4]]))
        assert_matches_oracle(case, out, lse, what=f"ragged S{S}")


def test_all_empty_batch():
    case = workloads.make_case("e", 2, 4, 2, 64, [0, 0], seed=401, pool_pages=2)
    out, lse, err, _ = run_gpu(case, max_context_len=16)
    assert err == 0
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ---- invariants
def test_single_token_is_v_row_bit_exact():
    case = workloads.make_case("one", 4, 16, 2, 256, [1, 1, 1, 1], seed=500, q_std=3.0)
    for S in (0, 16):
        case.partition_size = S
        out, lse, err, _ = run_gpu(case, max_context_len=16)
        assert err == 0
        for b in range(4):
            page = case.block_tables[b, 0]
            for h in range(16):
                vrow = case.v_cache[page, h // 8, 0].astype(np.float64)
                assert np.array_equal(out[b, h], vrow)
        ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                            case.context_lens, case.scale)
        assert np.abs(lse - ref[1]).max() <= 1e-4


def test_zero_query_gives_mean_of_v():
    case = workloads.make_case("q0", 2, 4, 2, 128, [777, 3000], seed=501)
    case.q[:] = 0
    out, lse, err, _ = run_gpu(case)
    assert err == 0
    for b, L in enumerate(case.context_lens):
        assert np.abs(lse[b] - math.log(L)).max() <= 1e-4
    assert_matches_oracle(case, out, lse, what="q=0")


def test_page_placement_is_bit_exact():
    case = workloads.make_case("perm", 2, 8, 2, 128, [1500, 999], seed=502)
    out1, lse1, _, _ = run_gpu(case)
    # Move every used page to a new physical slot and rewrite the table.
    rng = np.random.default_rng(7)
    perm = rng.permutation(case.num_pages).astype(np.int32)  # old -> new
    k2 = np.empty_like(case.k_cache)
    v2 = np.empty_like(case.v_cache)
    k2[perm] = case.k_cache
    v2[perm] = case.v_cache
    bt2 = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1)
    case2 = workloads.Case(**{**case.__dict__, "k_cache": k2, "v_cache": v2,
                              "block_tables": bt2.astype(np.int32)})
    out2, lse2, _, _ = run_gpu(case2)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_partition_count_invariance():
    case = workloads.make_case("pc", 2, 24, 4, 256, [20000, 7777], seed=503)
    ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                        case.context_lens, case.scale)
    outs = []
    for S in (16, 48, 512, 1024, 4096, 0):
        case.partition_size = S
        out, lse, err, _ = run_gpu(case)
        assert err == 0
        assert_matches_oracle(case, out, lse, ref=ref, what=f"S{S}")
        outs.append(out)
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() < 1e-2


def test_largest_partition_count():
    # 65 536 tokens in 16-token partitions: 4096 partitions per head, the most
    # the merge kernel reduces (16 chunks of 256).
    case = workloads.make_case("p4096", 1, 4, 1, 64, [65536], seed=504, partition_size=16)
    out, lse, err, plan = run_gpu(case)
    assert err == 0 and plan.num_partitions == 4096
    assert_matches_oracle(case, out, lse, what="4096 partitions")


def test_window_at_least_context_is_no_window():
    case = workloads.make_case("wl", 2, 8, 2, 64, [500, 64], seed=504)
    case.partition_size = 128
    a = run_gpu(case)
    case.window = 500
    b = run_gpu(case)
    case.window = 10 ** 6
    c = run_gpu(case)
    for x in (b, c):
        assert np.array_equal(a[0], x[0]) and np.array_equal(a[1], x[1])


def test_outputs_and_workspace_guards_untouched():
    case = workloads.make_case("guard", 3, 12, 4, 256, [5000, 33, 1200], seed=505)
    for S in (0, 512, 4096):
        case.partition_size = S
        out, lse, err, _ = run_gpu(case, guard=64)
        assert err == 0
        assert_matches_oracle(case, out, lse, what=f"guard S{S}")


def test_repeated_calls_reuse_workspace():
    case = workloads.make_case("rep", 2, 8, 2, 128, [900, 3000], seed=506)
    dev = to_device(case)
    a = run_gpu(case, dev=dev)
    b = run_gpu(case, dev=dev)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_max_shapes():
    # Largest head group per CTA (g = 8) and a two-chunk group (g = 16) at
    # D = 256, with the largest partition a CTA stages (256 pages).
    case = workloads.make_case("max", 2, 64, 4, 256, [4096, 4095], seed=507)
    for S in (4096, 0):
        case.partition_size = S
        out, lse, err, _ = run_gpu(case)
        assert err == 0
        assert_matches_oracle(case, out, lse, what=f"max S{S}")


def test_unwritten_slots_never_leak():
    """Cache slots outside the attended range (the tail of the last page, the
    head of the first page under a window) may hold anything, NaN included:
    they get weight 0 and must not reach the output."""
    lens = [37, 1000, 16, 3001]
    case = workloads.make_case("tail", len(lens), 8, 2, 128, lens, seed=508, window=700)
    ps = case.page_size
    for b, L in enumerate(lens):
        start = L - case.window if 0 < case.window < L else 0
        first, last = start // ps, (L - 1) // ps
        pf, pl = case.block_tables[b, first], case.block_tables[b, last]
        case.k_cache[pf, :, :start % ps] = np.float16(np.nan)
        case.v_cache[pf, :, :start % ps] = np.float16(np.nan)
        case.k_cache[pl, :, (L - 1) % ps + 1:] = np.float16(np.nan)
        case.v_cache[pl, :, (L - 1) % ps + 1:] = np.float16(np.inf)
    for S in (0, 64, 4096):
        case.partition_size = S
        out, lse, err, _ = run_gpu(case)
        assert err == 0
        assert_matches_oracle(case, out, lse, what=f"tail S{S}")


@pytest.mark.parametrize("ppc", [1, 2, 4])
def test_several_partitions_per_cta(ppc):
    """A CTA streaming several consecutive partitions (and merging them into
    one partial) gives the oracle's result, as one CTA per partition does;
    the CUDA-core kernel ignores the setting."""
    case = workloads.make_case("ppc", 3, 12, 2, 256, [20000, 7777, 1], seed=509, window=0)
    ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                        case.context_lens, case.scale)
    for S in (64, 512):
        case.partition_size = S
        out, lse, err, plan = run_gpu(case, guard=64, parts_per_cta=ppc)
        assert err == 0
        assert_matches_oracle(case, out, lse, ref=ref, what=f"ppc{ppc} S{S}")
    # one CTA (one partial) for all of a head's partitions: 2, 3 or 4
    # partitions of 32 tokens, and a sequence with a single partition
    scase = workloads.make_case("ppcs", 4, 8, 2, 128, [100, 70, 33, 20], seed=512, q_std=2.0)
    scase.partition_size = 32
    out, lse, err, plan = run_gpu(scase, guard=64, parts_per_cta=ppc)
    assert err == 0 and plan.num_partitions == 4
    assert_matches_oracle(scase, out, lse, what=f"ppc{ppc} one partial")
    wcase = workloads.make_case("ppcw", 2, 8, 4, 128, [9000, 3001], seed=510, window=2500)
    wcase.partition_size = 128
    out, lse, err, _ = run_gpu(wcase, parts_per_cta=ppc)
    assert err == 0
    assert_matches_oracle(wcase, out, lse, what=f"ppc{ppc} window")
    if gpu_helpers.KERNEL == "mma":
        # with the last-CTA merge: 8 partitions of 512 tokens, G x D/4 = 128 items
        fcase = workloads.make_case("ppcf", 3, 16, 4, 128, [4096, 1000, 2], seed=511)
        fcase.partition_size = 512
        out, lse, err, plan = run_gpu(fcase, guard=16, parts_per_cta=ppc, merge_in_kernel=1)
        assert err == 0 and plan.merge_in_kernel == 1 and plan.num_partitions == 8
        assert_matches_oracle(fcase, out, lse, what=f"ppc{ppc} last-CTA merge")


@pytest.mark.parametrize("fused", [0, 1])
def test_merge_in_kernel_and_merge_kernel_agree(fused):
    """The last-CTA merge inside the partition kernel and the separate merge
    kernel give the same result, with ragged, empty, unit and windowed
    sequences (the CUDA-core kernel always uses the merge kernel)."""
    lens = [0, 1, 4096, 17, 1000, 2, 3333]
    case = workloads.make_case("fm", len(lens), 16, 4, 128, lens, seed=511, window=1500)
    ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                        case.context_lens, case.scale, case.window)
    for S in (256, 512):  # 6 and 3 partitions: the in-kernel merge takes P <= 8
        case.partition_size = S
        out, lse, err, plan = run_gpu(case, guard=64, merge_in_kernel=fused)
        assert err == 0 and plan.num_partitions > 1
        assert_matches_oracle(case, out, lse, ref=ref, what=f"fused{fused} S{S}")


def test_workspace_reused_across_calls_and_shapes():
    """One workspace, several calls in a row with different inputs: the
    arrival counters and the error word come back to zero after each call."""
    a = workloads.make_case("wa", 3, 8, 2, 128, [900, 3000, 1], seed=512)
    b = workloads.make_case("wb", 3, 8, 2, 128, [2500, 40, 1700], seed=513)
    for c in (a, b):
        c.partition_size = 128
        c.block_tables = np.pad(c.block_tables, ((0, 0), (0, 200 - c.block_tables.shape[1])),
                                constant_values=-1)
    plan_probe = run_gpu(a, max_context_len=3200)[3]
    ws = torch.zeros(int(plan_probe.workspace_bytes), dtype=torch.uint8, device="cuda")
    for c in (a, b, a, b):
        out, lse, err, _ = run_gpu(c, max_context_len=3200, ws=ws)
        assert err == 0
        assert_matches_oracle(c, out, lse, what=c.name)


def _skip_d96_on_cuda_cores(D):
    if gpu_helpers.KERNEL == "simt" and D == 96:
        pytest.skip("the CUDA-core kernel is built for head dims 64/128/256")


@pytest.mark.parametrize("partition_size", [0, 16, 64, 512, 4096])
def test_head_dim_96(partition_size):
    _skip_d96_on_cuda_cores(96)
    case = workloads.make_case("d96", len(LENS), 12, 2, 96, LENS, seed=700,
                               partition_size=partition_size, q_std=2.0)
    out, lse, err, plan = run_gpu(case, guard=64)
    assert err == 0
    assert_matches_oracle(case, out, lse, what=f"D96 S{partition_size}")


@pytest.mark.parametrize("D", [64, 96, 128, 256])
@pytest.mark.parametrize("partition_size", [0, 64, 4096])
def test_bf16_cache(D, partition_size):
    _skip_d96_on_cuda_cores(D)
    case = workloads.make_case("bf16", len(LENS), 16, 4, D, LENS, seed=710 + D,
                               partition_size=partition_size, q_std=2.0, dtype="bf16")
    out, lse, err, plan = run_gpu(case, guard=64)
    assert err == 0
    rel = assert_matches_oracle(case, out, lse, what=f"bf16 D{D} S{partition_size}")
    print(f"bf16 D{D} S{partition_size}: rel L2 {rel:.2e}")


@pytest.mark.parametrize("dtype,D", [("bf16", 256), ("bf16", 96), ("f16", 96)])
def test_wider_paths_window_ragged_and_invariants(dtype, D):
    _skip_d96_on_cuda_cores(D)
    lens = [0, 1, 3001, 17, 5000]
    case = workloads.make_case("wide", len(lens), 8, 2, D, lens, seed=720 + D, window=1000,
                               q_std=3.0, dtype=dtype)
    # The in-kernel merge covers G x D/4 <= 128 items: not D = 256 with G = 4.
    for S, fused, ppc in ((0, None, None), (256, 1 if D < 256 else 0, None), (64, 0, 4)):
        case.partition_size = S
        out, lse, err, _ = run_gpu(case, guard=64, merge_in_kernel=fused, parts_per_cta=ppc)
        assert err == 0
        assert_matches_oracle(case, out, lse, what=f"{dtype} D{D} S{S}")
    # A single-token context returns that V row bit for bit.
    one = workloads.make_case("one", 3, 8, 2, D, [1, 1, 1], seed=721, dtype=dtype)
    out, lse, err, _ = run_gpu(one, max_context_len=16)
    for b in range(3):
        page = one.block_tables[b, 0]
        for h in range(8):
            row = one.v_cache[page, h // 4, 0]
            vals = (row.astype(np.uint32) << 16).view(np.float32) if dtype == "bf16" else row
            assert np.array_equal(out[b, h], vals.astype(np.float64))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 96, 128, 256])
@pytest.mark.parametrize("theta", [10000.0, 500000.0])
def test_rotary_embedding_in_kernel(D, theta, dtype):
    if gpu_helpers.KERNEL == "simt" and D == 96:
        pytest.skip("the CUDA-core kernel is built for head dims 64/128/256")
    case = workloads.make_case("rope", len(LENS), 8, 2, D, LENS, seed=800 + D, q_std=2.0,
                               rope_theta=theta, dtype=dtype)
    for S in (0, 64, 4096):
        case.partition_size = S
        out, lse, err, _ = run_gpu(case, guard=64)
        assert err == 0
        assert_matches_oracle(case, out, lse, what=f"rope D{D} S{S} {dtype}")
    # with a window, and positions past 2^16
    wcase = workloads.make_case("ropew", 2, 6, 2, D, [70000, 999], seed=801 + D, window=3000,
                                rope_theta=theta, dtype=dtype)
    out, lse, err, _ = run_gpu(wcase)
    assert err == 0
    assert_matches_oracle(wcase, out, lse, what=f"rope window D{D} {dtype}")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_fp32_cache(D):
    if gpu_helpers.KERNEL == "mma":
        pytest.skip("fp32 caches run on the CUDA-core kernel")
    case = workloads.make_case("f32", len(LENS), 12, 4, D, LENS, seed=900 + D, q_std=2.0,
                               dtype="f32")
    for S in (0, 64, 4096):
        case.partition_size = S
        out, lse, err, _ = run_gpu(case, guard=64)
        assert err == 0
        rel = assert_matches_oracle(case, out, lse, what=f"f32 D{D} S{S}")
        print(f"f32 D{D} S{S}: rel L2 {rel:.2e}")
    wcase = workloads.make_case("f32w", 3, 8, 2, D, [0, 5000, 333], seed=901 + D, window=700,
                                dtype="f32", rope_theta=10000.0)
    for S in (128, 4096):
        wcase.partition_size = S
        out, lse, err, _ = run_gpu(wcase, guard=64)
        assert err == 0
        assert_matches_oracle(wcase, out, lse, what=f"f32 rope window D{D} S{S}")


# ---- rotary embedding on the tensor-core kernel, over its plan shapes
ROPE_PLANS = {
    "one_partition": dict(partition_size=4096),
    "merge_kernel": dict(partition_size=96, cluster=False, merge_in_kernel=0),
    "two_per_cta": dict(partition_size=64, parts_per_cta=2, merge_in_kernel=0),
    "last_cta_merge": dict(partition_size=1024, merge_in_kernel=1),
    "cluster": dict(partition_size=256, cluster=True),
}


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("plan_kind", sorted(ROPE_PLANS))
@pytest.mark.parametrize("D,Hq,Hkv", [(64, 8, 2), (96, 12, 4), (128, 32, 8), (256, 8, 4)])
def test_rotary_tensor_core_plan_shapes(plan_kind, D, Hq, Hkv, dtype):
    if gpu_helpers.KERNEL != "mma":
        pytest.skip("tensor-core plan shapes")
    kw = dict(ROPE_PLANS[plan_kind])
    lens = [1, 17, 700, 2049, 3333]
    case = workloads.make_case("ropep", len(lens), Hq, Hkv, D, lens, seed=1600 + D, q_std=2.0,
                               rope_theta=500000.0, window=3000 if plan_kind == "cluster" else 0,
                               dtype=dtype)
    out, lse, err, plan = run_gpu(case, guard=16, **kw)
    assert err == 0 and plan.kernel == 2 and plan.rope_theta > 0
    assert_matches_oracle(case, out, lse, what=f"rope mma {plan_kind} D{D} {dtype}")
