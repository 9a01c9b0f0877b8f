"""rk_seg_attn_forward_host: the forward with q, out and lse in host memory
(copies overlapped with the kernels) gives the device forward's results bit
for bit, for every prefill kernel and for decode."""
import numpy as np
import pytest
import torch

from _helpers import compare, oracle_rows, run_gpu, sample_rows
from position_independent_kv_gb300 import binding as B
from position_independent_kv_gb300 import build as BUILD
from position_independent_kv_gb300.protected import build_bitmap
from position_independent_kv_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu

KERNELS = {"default": 0, "cta_pair": B.RK_PLAN_CTA_PAIR, "single_cta": B.RK_PLAN_SINGLE_CTA,
           "legacy": B.RK_PLAN_LEGACY_MMA}


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BUILD.build()


def _host_forward(wl, flags, pinned=True):
    bm, _ = build_bitmap(wl)
    plan = B.SegAttnPlan.from_workload(wl, bitmap=bm, flags=flags)
    ws = None
    if plan.workspace_bytes:
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=wl.q.device)
    hq = torch.empty(wl.q.shape, dtype=wl.q.dtype, pin_memory=pinned)
    ho = torch.empty(wl.out_init.shape, dtype=wl.out_init.dtype, pin_memory=pinned)
    hl = torch.empty(wl.lse_init.shape, dtype=wl.lse_init.dtype, pin_memory=pinned)
    hq.copy_(wl.q)
    ho.copy_(wl.out_init)
    hl.copy_(wl.lse_init)
    # device buffers hold stale values: the call must overwrite them from the host
    dq = torch.zeros_like(wl.q)
    do = torch.full_like(wl.out_init, 7.0)
    dl = torch.full_like(wl.lse_init, -3.0)
    plan.forward_host(hq, ho, hl, dq, do, dl, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    return ho, hl, plan


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("name", ["tiny", "flash_mini", "ctx128k_mini", "decode_mini", "ctx16k"])
def test_host_forward_matches_device_forward(name, kernel):
    wl = make_workload(name, seed=0, device="cuda", q_scale=4.0)
    out, lse, plan, _, _ = run_gpu(wl, flags=KERNELS[kernel])
    ho, hl, plan2 = _host_forward(wl, KERNELS[kernel])
    assert torch.equal(ho, out.cpu()), "out differs from the device forward"
    assert torch.equal(hl, lse.cpu()), "lse differs from the device forward"
    plan.close()
    plan2.close()


def test_host_forward_pageable_memory():
    wl = make_workload("flash_mini", seed=1, device="cuda")
    out, lse, plan, _, _ = run_gpu(wl)
    ho, hl, plan2 = _host_forward(wl, 0, pinned=False)
    assert torch.equal(ho, out.cpu()) and torch.equal(hl, lse.cpu())
    plan.close()
    plan2.close()


# Global head sets other than one head per group of eight: three runs of
# consecutive heads (one strided copy per run comes back) and every fourth
# head (one strided copy per row range); five Global heads also tile the
# 128 query pairs of a Global tile unevenly (25 rows x 5 heads)
ROLES = {"runs": [0, 1, 2, 9, 33], "stride4": list(range(1, 64, 4))}


@pytest.mark.parametrize("roles", list(ROLES))
@pytest.mark.parametrize("kernel", ["default", "cta_pair"])
def test_host_forward_other_global_heads(roles, kernel):
    wl = make_workload("flash_mini", seed=2, device="cuda", q_scale=4.0)
    role = np.zeros(wl.H, np.uint8)
    role[ROLES[roles]] = 1
    wl.head_role = role
    out, lse, plan, _, prot_rows = run_gpu(wl, flags=KERNELS[kernel])
    rng = np.random.default_rng(5)
    rows = [sample_rows(req, prot_rows[r], rng, wl.window, wl.sink, cap=24)
            for r, req in enumerate(wl.requests)]
    compare(wl, out, lse, prot_rows, oracle_rows(wl, prot_rows, rows), rows, label=roles)
    ho, hl, plan2 = _host_forward(wl, KERNELS[kernel])
    assert torch.equal(ho, out.cpu()), "out differs from the device forward"
    assert torch.equal(hl, lse.cpu()), "lse differs from the device forward"
    plan.close()
    plan2.close()
