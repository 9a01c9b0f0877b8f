"""rk_protected_build (the protected-row set on the device) against the
oracle's builder, bit for bit, on every workload's geometry and on edge
rules; and a plan fed the device bitmap gives the same forward."""
import numpy as np
import pytest
import torch

import oracle as O
from _helpers import run_gpu
from position_independent_kv_gb300 import binding as B
from position_independent_kv_gb300 import build as BUILD
from position_independent_kv_gb300.protected import build_bitmap
from position_independent_kv_gb300.workloads import make_geometry, make_workload

pytestmark = pytest.mark.gpu

NAMES = ["tiny", "flash", "varlen", "ctx128k", "decode", "flash_mini", "varlen_mini",
         "ctx128k_mini", "decode_mini"]


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BUILD.build()


def _score_from_perm(perm):
    """Scores whose descending order is the permutation (no ties)."""
    s = np.empty(len(perm), np.float32)
    s[perm] = -np.arange(len(perm), dtype=np.float32)
    return s


def _device_bitmap(wl, boundary, p_random, budget_pct, none, scores, dirty_rows=None):
    segs, begins = [], [0]
    for r in wl.requests:
        segs += [(s.n, s.delta, s.is_new) for s in r.segments]
        begins.append(len(segs))
    u = torch.from_numpy(np.concatenate([r.u for r in wl.requests]).astype(np.float64)).cuda()
    sc = torch.from_numpy(np.concatenate(scores).astype(np.float32)).cuda()
    nwords = sum((r.T + 31) // 32 for r in wl.requests)
    dirty = None
    if dirty_rows is not None:
        dirty = torch.from_numpy(np.concatenate([O.bitmap_words(d) for d in dirty_rows])
                                 .view(np.int32)).cuda()
    bitmap = torch.full((nwords,), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.protected_workspace_bytes(len(wl.requests), len(segs)), dtype=torch.uint8,
                     device="cuda")
    B.protected_build(segs, begins, boundary, p_random, budget_pct, none, u, sc, dirty, bitmap, ws)
    torch.cuda.synchronize()
    return bitmap.cpu().numpy().view(np.uint32)


def _oracle_bitmap(wl, boundary, p_random, budget_pct, none, perms, dirty_rows=None):
    words = []
    for i, r in enumerate(wl.requests):
        segs = [(s.n, s.delta, s.is_new) for s in r.segments]
        prot = O.build_protected(r.T, segs, boundary, p_random, budget_pct / 100.0, none, r.u,
                                 perms[i], dirty=None if dirty_rows is None else dirty_rows[i])
        words.append(O.bitmap_words(prot))
    return np.concatenate(words)


@pytest.mark.parametrize("name", NAMES)
def test_device_builder_matches_oracle(name):
    wl = make_geometry(name, 0)
    r = wl.rule
    pct = int(round(100 * r.budget))
    scores = [_score_from_perm(q.perm) for q in wl.requests]
    got = _device_bitmap(wl, r.boundary, r.p_random, pct, r.none, scores)
    want = _oracle_bitmap(wl, r.boundary, r.p_random, pct, r.none, [q.perm for q in wl.requests])
    assert np.array_equal(got, want)
    # and the host builder of the workloads agrees too
    host, _ = build_bitmap(wl)
    assert np.array_equal(got, host)


@pytest.mark.parametrize("rule", ["budget_ties", "budget_100", "bernoulli_all", "boundary_huge",
                                  "none_dirty", "budget_dirty"])
def test_device_builder_edge_rules(rule):
    wl = make_geometry("varlen_mini", 0)
    rng = np.random.default_rng(11)
    perms, scores, dirty = [], [], None
    for q in wl.requests:
        # few distinct scores: ties are broken by the lower row first
        s = np.floor(rng.random(q.T) * 7).astype(np.float32) - 3.0
        s[rng.random(q.T) < 0.1] = -0.0
        scores.append(s)
        rows = np.arange(q.T)
        perms.append(np.lexsort((rows, -s.astype(np.float64))))
    if rule in ("none_dirty", "budget_dirty"):
        dirty = [rng.random(q.T) < 0.07 for q in wl.requests]
    args = {"budget_ties": (24, 0.0, 20, False), "budget_100": (24, 0.0, 100, False),
            "bernoulli_all": (24, 1.0, 0, False), "boundary_huge": (100000, 0.0, 25, False),
            "none_dirty": (24, 0.0, 25, True), "budget_dirty": (5, 0.0, 25, False)}[rule]
    got = _device_bitmap(wl, *args, scores, dirty)
    want = _oracle_bitmap(wl, *args, perms, dirty)
    assert np.array_equal(got, want)


def test_plan_takes_the_device_bitmap():
    wl = make_workload("ctx128k_mini", seed=2, device="cuda")
    r = wl.rule
    scores = [_score_from_perm(q.perm) for q in wl.requests]
    bits = _device_bitmap(wl, r.boundary, r.p_random, int(round(100 * r.budget)), r.none, scores)
    out_h, lse_h, plan, _, _ = run_gpu(wl)
    d_bits = torch.from_numpy(bits.view(np.int32)).cuda()
    plan2 = B.SegAttnPlan.from_workload(wl, bitmap=d_bits, flags=B.RK_PLAN_DEVICE_BITMAP)
    out = wl.out_init.clone()
    lse = wl.lse_init.clone()
    ws = torch.empty(max(16, plan2.workspace_bytes), dtype=torch.uint8, device="cuda")
    plan2.forward(wl.q, out, lse, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, out_h) and torch.equal(lse, lse_h)
    assert plan2.info["protected_local_rows"] == plan.info["protected_local_rows"]
    plan.close()
    plan2.close()
