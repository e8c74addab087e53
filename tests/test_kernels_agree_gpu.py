"""The two partition kernels agree with each other.

apache/tvm PR #20426 (section Correctness) checks its two decode nests against
each other as well as against the f64 reference.  Here the tensor-core kernel
and the CUDA-core kernel run on identical inputs -- plain, windowed, bf16 and
rotary cases over context lengths 1 .. 3060 with a shuffled page table -- and
their outputs and LSEs are compared directly, besides each matching the fp64
oracle.  The two differ in arithmetic only (the tensor-core kernel rounds the
softmax weights to the cache type for P.V), so they agree well inside the
parity bar."""
import numpy as np
import pytest

import gpu_helpers
import oracle
from gpu_helpers import assert_matches_oracle, rel_l2, run_gpu
from paged_kv_gqa_pa_gb300 import workloads

pytestmark = pytest.mark.gpu

LENS = [1, 15, 16, 17, 255, 257, 513, 3060]


def _both(case, **kw):
    res = {}
    for kernel in ("mma", "simt"):
        gpu_helpers.KERNEL = kernel
        try:
            out, lse, err, plan = run_gpu(case, **kw)
        finally:
            gpu_helpers.KERNEL = None
        assert err == 0
        res[kernel] = (out, lse)
    return res


@pytest.mark.parametrize("D,Hq,Hkv,dtype,window,theta", [
    (64, 8, 2, "f16", 0, 0.0),
    (128, 32, 8, "f16", 0, 0.0),
    (256, 24, 4, "f16", 1000, 0.0),
    (128, 16, 4, "bf16", 0, 0.0),
    (128, 8, 2, "f16", 0, 10000.0),
    (64, 8, 2, "bf16", 700, 500000.0),
])
def test_tensor_core_and_cuda_core_kernels_agree(D, Hq, Hkv, dtype, window, theta):
    case = workloads.make_case("agree", len(LENS), Hq, Hkv, D, LENS, seed=1800 + D, q_std=2.0,
                               window=window, dtype=dtype, rope_theta=theta)
    ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
                        case.scale, case.window, dtype=case.dtype, rope_theta=case.rope_theta)
    for S in (0, 64):
        case.partition_size = S
        res = _both(case)
        (om, lm), (os_, ls) = res["mma"], res["simt"]
        for o, l, k in ((om, lm, "mma"), (os_, ls, "simt")):
            assert_matches_oracle(case, o, l, ref=ref, what=f"{k} D{D} {dtype} S{S}")
        # against each other: within the parity bar, and both LSEs finite in the same places
        bar = gpu_helpers.REL_L2_TOL_BF16 if dtype == "bf16" else gpu_helpers.REL_L2_TOL
        assert rel_l2(om, os_) <= bar
        assert np.array_equal(np.isfinite(lm), np.isfinite(ls))
        fin = np.isfinite(lm)
        assert np.abs(lm[fin] - ls[fin]).max() <= gpu_helpers.LSE_TOL


@pytest.mark.parametrize("dtype,theta", [("f16", 0.0), ("bf16", 0.0), ("f32", 0.0),
                                         ("f16", 10000.0), ("bf16", 10000.0)])
def test_convenience_decode_follows_q_dtype(dtype, theta):
    # binding.decode plans, allocates and decodes in one call; the element
    # type comes from q.
    import torch
    import paged_kv_gqa_pa_gb300 as pa
    case = workloads.make_case("conv", 3, 8, 2, 128, [1, 700, 3060], seed=1900, window=1500,
                               dtype=dtype, rope_theta=theta)
    dev = gpu_helpers.to_device(case)
    out, lse, plan, err = pa.decode(dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"],
                                    case.scale, window=case.window, rope_theta=theta)
    assert err == 0 and out.dtype == dev["q"].dtype and plan.rope_theta == theta
    assert_matches_oracle(case, out.double().cpu().numpy(), lse.double().cpu().numpy(),
                          what=f"decode() {dtype} theta {theta}")
