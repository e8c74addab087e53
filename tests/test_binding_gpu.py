"""The Python binding's prepared call: pa_decode's arguments checked and
converted once, then the C call alone per step.  It must give exactly what
pa_decode gives on the same plan (the same kernels), follow new contents of
the same buffers, and keep the plan it was prepared with."""
import numpy as np
import pytest
import torch

import paged_kv_gqa_pa_gb300 as pa
from gpu_helpers import assert_matches_oracle, ensure_built, to_device
from paged_kv_gqa_pa_gb300 import workloads

pytestmark = pytest.mark.gpu


def test_prepared_call_matches_pa_decode_and_follows_the_inputs():
    ensure_built()
    cases = [workloads.make_case("prep", 3, 16, 4, 128, [900 + i, 2500 - i, 33 + i], seed=2200 + i,
                                 pool_pages=500, max_pages_per_seq=200) for i in range(2)]
    c0 = cases[0]
    B, Hq, D = c0.q.shape
    plan = pa.pa_plan_ex(B, Hq, c0.Hkv, D, 16, c0.num_pages, c0.max_pages_per_seq, 3200, 0, 0,
                         torch.cuda.get_device_properties(0).multi_processor_count)
    dev = to_device(c0)
    out = torch.empty((B, Hq, D), dtype=torch.float16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    ws = pa.new_workspace(plan, "cuda")
    call = pa.prepare_decode(plan, dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"], c0.scale, 0,
                             out, lse, ws)
    plan.kernel = 99  # the prepared call keeps its own copy of the plan
    for c in cases:
        new = to_device(c)
        for name in ("q", "k", "v", "bt", "cl"):
            dev[name].copy_(new[name])
        call()
        torch.cuda.synchronize()
        got = (out.clone(), lse.clone())
        ref_plan = pa.pa_plan_ex(B, Hq, c0.Hkv, D, 16, c0.num_pages, c0.max_pages_per_seq, 3200,
                                 0, 0, torch.cuda.get_device_properties(0).multi_processor_count)
        pa.pa_decode(ref_plan, dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"], c.scale, 0,
                     out, lse, ws)
        torch.cuda.synchronize()
        assert torch.equal(got[0].view(torch.int16), out.view(torch.int16))
        assert torch.equal(got[1].view(torch.int32), lse.view(torch.int32))
        assert pa.pa_get_error(ws) == 0
        assert_matches_oracle(c, got[0].double().cpu().numpy(), got[1].double().cpu().numpy(),
                              what="prepared call")
