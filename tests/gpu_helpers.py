"""Shared helpers of the GPU tests: upload a seeded case, run the CUDA path
through the C ABI, compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_gqa_pa_gb300 as pa
from paged_kv_gqa_pa_gb300 import build as pa_build

# Tolerances: relative L2 over the whole output tensor, absolute on the LSE.
# fp16 output: 1e-3.  bf16 output: its rounding alone (unit roundoff 2^-9)
# gives a relative L2 near 2^-9/sqrt(3) = 1.1e-3, so the bar is 3e-3.
REL_L2_TOL = 1e-3
REL_L2_TOL_BF16 = 3e-3
# fp32 output: no output rounding; exp2 approximation (2^-22) and fp32 sums.
REL_L2_TOL_F32 = 1e-4
LSE_TOL = 1e-4

_built = False

# Partition-kernel variant the GPU tests run (set per test by a fixture);
# None keeps the planner's choice.
KERNEL = None
KERNELS = {"mma": 2, "simt": 1}


def ensure_built():
    global _built
    if not _built:
        pa_build.build()
        _built = True
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pa.load()


def _elems(a, dtype):
    t = torch.from_numpy(a)
    return t.view(torch.bfloat16) if dtype == "bf16" else t


def to_device(case, device="cuda"):
    return dict(
        q=_elems(case.q, case.dtype).to(device),
        k=_elems(case.k_cache, case.dtype).to(device),
        v=_elems(case.v_cache, case.dtype).to(device),
        bt=torch.from_numpy(case.block_tables).to(device),
        cl=torch.from_numpy(case.context_lens).to(device),
    )


def run_gpu(case, partition_size=None, max_context_len=None, dev=None, num_sms=None,
            guard=0, parts_per_cta=None, merge_in_kernel=None, ws=None, cluster=None,
            prewait_prefetch=None, test_stall_bytes=None, deep_ring=None):
    """Plan + pa_decode through the C ABI.  Returns (out fp64 numpy, lse fp64
    numpy, device error word, plan).  With guard > 0 the outputs and the
    workspace sit inside larger NaN/0xA5-filled buffers whose guard regions are
    checked afterwards.  cluster: True forces the cluster merge (the plan's
    partition count must be 2..16), False forbids it, None keeps the planner's
    choice; forcing several partitions per CTA or the last-CTA merge drops it.
    prewait_prefetch overrides the plan's pre-wait L2 prefetch (pages per warp);
    test_stall_bytes sets the plan's copy-timeout test hook; deep_ring picks
    the cluster instance with deeper page rings (1) or not (0)."""
    ensure_built()
    dev = dev or to_device(case)
    B, Hq, D = case.q.shape
    if partition_size is None:
        partition_size = case.partition_size
    if max_context_len is None:
        max_context_len = max(case.max_context_len, 0)
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = pa.pa_plan_ex(B, Hq, case.Hkv, D, case.page_size, case.num_pages,
                         case.max_pages_per_seq, max_context_len, case.window, partition_size,
                         num_sms, dtype={"f16": 0, "bf16": 1, "f32": 2}[case.dtype],
                         kernel=KERNELS[KERNEL] if KERNEL is not None else 0,
                         rope_theta=case.rope_theta)
    if parts_per_cta is not None:
        plan.parts_per_cta = parts_per_cta
        if parts_per_cta > 1:
            plan.cluster = 0
    if merge_in_kernel is not None:
        plan.merge_in_kernel = merge_in_kernel
        if merge_in_kernel:
            plan.cluster = 0
    if cluster is True:
        assert 2 <= plan.num_partitions <= 16, plan.num_partitions
        plan.cluster = plan.num_partitions
        plan.parts_per_cta = 1
        plan.merge_in_kernel = 0
    elif cluster is False:
        plan.cluster = 0
    if prewait_prefetch is not None:
        plan.prewait_prefetch = prewait_prefetch
    if test_stall_bytes is not None:
        plan.test_stall_bytes = test_stall_bytes
    if deep_ring is not None:
        plan.deep_ring = deep_ring
    n_out = B * Hq * D
    et = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[case.dtype]
    out_buf = torch.full((n_out + 2 * guard,), float("nan"), dtype=et, device="cuda")
    lse_buf = torch.full((B * Hq + 2 * guard,), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = int(plan.workspace_bytes)
    out = out_buf[guard:guard + n_out].view(B, Hq, D)
    lse = lse_buf[guard:guard + B * Hq].view(B, Hq)
    if ws is None:
        # Only the control bytes start at zero; the partials area holds junk
        # (0xA5), so nothing may rely on it being cleared.
        ws_buf = torch.full((ws_bytes + 2 * guard * 16,), 0xA5, dtype=torch.uint8, device="cuda")
        ws = ws_buf[guard * 16:guard * 16 + ws_bytes]
        ws[:plan.ctrl_bytes].zero_()
    else:
        ws_buf = None
        assert ws.numel() >= ws_bytes
    pa.pa_decode(plan, dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"], case.scale,
                 case.window, out, lse, ws)
    err = pa.pa_get_error_ex(ws, clear=True)
    torch.cuda.synchronize()
    # Every call leaves the control bytes (error word, arrival counters) zero.
    assert int(ws[:plan.ctrl_bytes].count_nonzero()) == 0, "control bytes not left zero"
    if guard and ws_buf is not None:
        ob = out_buf.cpu()
        lb = lse_buf.cpu()
        wb = ws_buf.cpu()
        assert torch.isnan(ob[:guard]).all() and torch.isnan(ob[guard + n_out:]).all(), "out guard"
        assert torch.isnan(lb[:guard]).all() and torch.isnan(lb[guard + B * Hq:]).all(), "lse guard"
        assert (wb[:guard * 16] == 0xA5).all() and (wb[guard * 16 + ws_bytes:] == 0xA5).all(), \
            "workspace guard"
    return (out.double().cpu().numpy(), lse.double().cpu().numpy(), err, plan)


def rel_l2(a, b):
    den = np.linalg.norm(b.ravel())
    num = np.linalg.norm((a - b).ravel())
    return num / den if den > 0 else num


def assert_matches_oracle(case, out, lse, ref=None, what=""):
    if ref is None:
        ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                            case.context_lens, case.scale, case.window, dtype=case.dtype,
                            rope_theta=case.rope_theta)
    ref_out, ref_lse = ref
    assert not np.isnan(out).any(), f"{what}: NaN in output"
    err = rel_l2(out, ref_out)
    tol = {"bf16": REL_L2_TOL_BF16, "f32": REL_L2_TOL_F32}.get(case.dtype, REL_L2_TOL)
    assert err <= tol, f"{what}: rel L2 {err:.3e} > {tol}"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: LSE finiteness differs"
    assert np.array_equal(lse[~fin], ref_lse[~fin]), f"{what}: LSE of empty rows"
    if fin.any():
        d = np.abs(lse[fin] - ref_lse[fin]).max()
        assert d <= LSE_TOL, f"{what}: |dLSE| {d:.3e} > {LSE_TOL}"
    return err
