"""pa_decode captured once in a CUDA graph and replayed with new inputs.

A decode loop captures its step once and replays it every token: the K/V
pools, the block table, the lengths, q and the outputs stay at the same
addresses while their contents change between replays.  Every plan kind must
give the fp64 oracle's result on each replay, for the inputs in place at that
replay: the lengths and page ids are read by the kernels, never baked into
the launch, and the arrival counters of the last-CTA merge are back at zero
after every replay.  Each case replays three steps whose lengths grow by one
token per step (a decode step's new token), with a page table reshuffled in
between."""
import numpy as np
import pytest
import torch

import gpu_helpers
import paged_kv_gqa_pa_gb300 as pa
from gpu_helpers import assert_matches_oracle, ensure_built, to_device
from paged_kv_gqa_pa_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

# (partition_size, plan edits) per plan kind; the lengths of the case give
# each its shape.
KINDS = {
    "unsplit": (4096, {}),
    "merge_kernel": (96, dict(cluster=0, merge_in_kernel=0)),
    "last_cta_merge": (256, dict(cluster=0, merge_in_kernel=1)),
    "cluster": (256, "cluster"),
    "balanced": (binding.PA_PARTITION_BALANCED, {}),
}


def _step_case(lens, seed, window):
    return workloads.make_case("graph", len(lens), 16, 4, 128, lens, seed=seed, window=window,
                               max_pages_per_seq=260, pool_pages=1200)


@pytest.mark.parametrize("window", [0, 700])
@pytest.mark.parametrize("kind", sorted(KINDS))
def test_graph_replays_follow_the_inputs(kind, window):
    ensure_built()
    base = [3000, 1200, 2049, 77]
    # Three decode steps: every length one token longer than the step before,
    # each step with its own values and its own page placement (same pool).
    steps = [_step_case([L + i for L in base], 2100 + i, window) for i in range(3)]
    S, edits = KINDS[kind]
    c0 = steps[0]
    B, Hq, D = c0.q.shape
    max_len = 4096
    plan = pa.pa_plan_ex(B, Hq, c0.Hkv, D, 16, c0.num_pages, c0.max_pages_per_seq, max_len, window,
                         S, torch.cuda.get_device_properties(0).multi_processor_count)
    if edits == "cluster":
        assert 2 <= plan.num_partitions <= 16
        plan.cluster, plan.parts_per_cta, plan.merge_in_kernel = plan.num_partitions, 1, 0
    else:
        for k, v in edits.items():
            setattr(plan, k, v)
    if kind == "balanced":
        assert plan.balanced > 0
    dev = to_device(c0)
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = pa.new_workspace(plan, "cuda")

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        pa.pa_decode(plan, dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"], c0.scale, window,
                     out, lse, ws, stream)  # warm-up outside the capture
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            pa.pa_decode(plan, dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"], c0.scale,
                         window, out, lse, ws, stream)
    for i, c in enumerate(steps):
        # new contents at the captured addresses
        host = to_device(c)
        for name in ("q", "k", "v", "bt", "cl"):
            dev[name].copy_(host[name])
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert pa.pa_get_error(ws) == 0, f"replay {i}"
        ctrl = ws[:plan.ctrl_bytes]
        assert int(ctrl.count_nonzero()) == 0, f"replay {i}: control bytes not left zero"
        assert_matches_oracle(c, out.double().cpu().numpy(), lse.double().cpu().numpy(),
                              what=f"graph replay {i}, {kind}, window {window}")
