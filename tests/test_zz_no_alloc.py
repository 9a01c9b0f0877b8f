"""rk_seg_attn_forward_noalloc, the forward for callers that cannot allocate
device memory when they issue it (engines that reserve all memory up front).
It keeps the split-over-segments scratch in the library's static device
array; its results must match rk_seg_attn_forward with a caller workspace,
bit for bit, on two calls in a row (the array keeps the previous call's
contents).  Both entry points run the same kernels on the same plan and the
split merge adds its parts in a fixed order, so any difference would be a
scratch-layout or clearing mistake.

This file is collected last on purpose."""
import math

import numpy as np
import pytest
import torch

from position_independent_kv_gb300 import binding as B
from position_independent_kv_gb300 import build as BUILD
from position_independent_kv_gb300.protected import build_bitmap
from position_independent_kv_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BUILD.build()


@pytest.mark.parametrize("name", ["decode_mini", "decode"])
def test_noalloc_matches_workspace_forward(name):
    wl = make_workload(name, seed=4, device="cuda", q_scale=2304.0)
    bm, prot = build_bitmap(wl)
    plan = B.SegAttnPlan.from_workload(wl, bitmap=bm)
    assert 0 < plan.workspace_bytes <= (32 << 20)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    r_out, r_lse = wl.out_init.clone(), wl.lse_init.clone()
    plan.forward(wl.q, r_out, r_lse, ws)
    torch.cuda.synchronize()
    for call in range(2):
        out, lse = wl.out_init.clone(), wl.lse_init.clone()
        plan.forward_noalloc(wl.q, out, lse)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert torch.equal(out, r_out), f"call {call}: out differs"
        assert torch.equal(lse, r_lse), f"call {call}: lse differs"


def test_noalloc_refuses_oversized_scratch():
    """A plan whose scratch exceeds the static array is refused before any
    launch; the outputs keep their bytes."""
    R, n, H = 600, 4096, 64
    lat = (torch.randn(n, 576, device="cuda") / 24).to(torch.bfloat16)
    new = (torch.randn(R, 576, device="cuda") / 24).to(torch.bfloat16)
    segs, begins = [], [0]
    for r in range(R):
        segs += [(lat, n, 0, False), (new[r], 1, n, True)]
        begins.append(len(segs))
    role = np.zeros(H, np.uint8)
    role[7::8] = 1
    plan = B.SegAttnPlan(segs, begins, [n] * R, H, 512, 64, 10000.0, 1 / math.sqrt(576),
                         role, 4, 256)
    assert plan.workspace_bytes > (32 << 20)
    q = (torch.randn(R, H, 576, device="cuda") / 24).to(torch.bfloat16)
    out = torch.zeros(R, H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((R, H), 3.0, device="cuda")
    with pytest.raises(B.RkError) as ei:
        plan.forward_noalloc(q, out, lse)
    assert ei.value.status == 6
    torch.cuda.synchronize()
    assert bool((out == 0).all()) and bool((lse == 3.0).all())
