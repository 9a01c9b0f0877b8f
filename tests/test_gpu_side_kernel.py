"""The side kernel beside the 4-CTA clusters: a persistent CTA-pair kernel on
the SMs that 4-CTA clusters leave free takes the shortest tile pairs from the
back of the work queue.  It computes each pair with the 4-CTA kernel's
arithmetic (the same score chain order, the shared online softmax, the same
P.V order and epilogue), so a forward's outputs and LSEs must be bit for bit
the ones of the same plan with RK_PLAN_NO_SIDE_PAIRS, whichever pairs the side
kernel happened to take.  The oracle comparisons of the default path are in
the parity tests; this file checks the identity and that the side kernel did
take pairs."""
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


def _forward(wl, bm, flags):
    plan = B.SegAttnPlan.from_workload(wl, bitmap=bm, flags=flags)
    assert plan.info["kernel"] == 3
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    out, lse = wl.out_init.clone(), wl.lse_init.clone()
    for _ in range(2):  # the second forward's queue is read below
        plan.forward(wl.q, out, lse, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    # a prefill-only plan keeps its work queue at the start of the workspace:
    # a 64-bit counter of pairs taken from the front (low half) and claims
    # made from the back (high half)
    word = int(ws[:8].cpu().view(torch.int64).item()) & ((1 << 64) - 1)
    info = plan.info
    plan.close()
    return out, lse, word >> 32, info


@pytest.mark.parametrize("name,sharp", [("ctx16k", False), ("ctx128k_mini", True),
                                        ("flash_mini", False), ("varlen_mini", True),
                                        ("edge_many_segs", False),
                                        ("ctx128k_vrope_mini", True), ("flash_vrope_mini", False)])
def test_side_kernel_is_bit_identical(name, sharp):
    wl = make_workload(name, seed=1, device="cuda")
    if sharp:  # score std ~4: q scaled by 4 d_k
        wl = make_workload(name, seed=1, device="cuda", q_scale=4.0 * (wl.d_nope + wl.d_rope))
    bm, _ = build_bitmap(wl)
    out_s, lse_s, back_s, info_s = _forward(wl, bm, 0)
    out_n, lse_n, back_n, info_n = _forward(wl, bm, B.RK_PLAN_NO_SIDE_PAIRS)
    assert info_s["side_pairs"] > 0 and info_n["side_pairs"] == 0
    assert back_n == 0, "no claims from the back with RK_PLAN_NO_SIDE_PAIRS"
    def diff(x, y):
        d = (x.float() - y.float()).abs()
        return f"{int((x != y).sum())} of {x.numel()} differ, max {float(d.max()):.3g}"
    assert torch.equal(out_s, out_n), f"{name}: outputs differ with the side kernel: {diff(out_s, out_n)}"
    assert torch.equal(lse_s, lse_n), f"{name}: LSEs differ with the side kernel: {diff(lse_s, lse_n)}"
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if name == "ctx16k" and sms == 152:
        # 36 clusters of 4 leave 8 SMs: 4 side CTA pairs, each of which ends
        # with one failed claim; more claims than that took pairs
        assert back_s > 4, f"the side kernel took no pair ({back_s} claims)"
