"""Host logic of the 4-CTA prefill kernel's work list, checked on host-only
plans against the segment geometry: every tile lies in exactly one pair, a
pair's key ranges cover those of its tiles, pairs come longest first, and the
segment-skip hint of a pair names only segments that meet neither of its key
ranges (the key walk jumps over them without reading their offsets)."""
from __future__ import annotations

import numpy as np
import pytest

from position_independent_kv_gb300 import binding as B
from position_independent_kv_gb300.protected import build_bitmap
from position_independent_kv_gb300.workloads import make_geometry, segments_for_abi

TN = 128  # keys per key tile


def _host_plan(name):
    wl = make_geometry(name, 0)
    bm, _ = build_bitmap(wl)
    flat, begins = segments_for_abi(wl)
    segs = [(0x10000000 + i * 0x1000000, s[1], s[2], s[3]) for i, s in enumerate(flat)]
    plan = B.SegAttnPlan(segments=segs, seg_begin=begins,
                         q_row_begin=[r.q_row_begin for r in wl.requests], num_heads=wl.H,
                         d_nope=wl.d_nope, d_rope=wl.d_rope, rope_base=wl.rope_base,
                         softmax_scale=wl.scale, head_role=wl.head_role, sink=wl.sink,
                         window=wl.window, bitmap=bm,
                         flags=B.RK_PLAN_HOST_ONLY | (B.RK_PLAN_V_ROPE if wl.v_rope else 0))
    return wl, plan


def _segments(wl, r):
    """(delta, n) of request r's segments, sorted by offset (the plan's order)."""
    return sorted((int(s.delta), int(s.n)) for s in wl.requests[r].segments)


def _walk_tiles(segs, sh, wl_, kh):
    """Key tiles of the walk over [0, sh) u [wl_, kh), segment by segment."""
    n = 0
    for d, ln in segs:
        for lo, hi in ((0, sh), (wl_, kh)):
            a, b = max(lo, d), min(hi, d + ln)
            if a < b:
                n += -(-(b - a) // TN)
    return n


def _inside(a0, a1, b0, b1):
    """[a0, a1) lies inside [b0, b1) (empty ranges lie anywhere)."""
    return a0 >= a1 or (b0 <= a0 and a1 <= b1)


@pytest.mark.parametrize("name", ["ctx16k", "varlen_mini", "flash_mini", "ctx128k_mini",
                                  "edge_many_segs", "ctx128k_vrope_mini", "decode_vrope_mini"])
def test_pairs_cover_tiles_and_skip_only_unneeded_segments(name):
    wl, plan = _host_plan(name)
    if plan.info["kernel"] != 3:
        pytest.skip("not on the 4-CTA kernel")
    pr = plan.pairs()
    assert pr.shape[0] > 0
    real = 0
    costs = []
    skipped_any = False
    for rec in pr:
        t = [rec[0:8], rec[8:16]]
        kh, wl_, sh = int(rec[16]), int(rec[17]), int(rec[18])
        skip = int(rec[19]) & 0xffffffff
        assert t[0][0] == t[1][0], "both tiles of a pair belong to one request"
        assert t[0][7] & 1 == 0, "the first tile of a pair does work"
        assert sh <= wl_ <= kh
        r = int(t[0][0])
        segs = _segments(wl, r)
        for tile in t:
            if tile[7] & 1:
                continue
            real += 1
            tkh, twl, tsh = int(tile[4]), int(tile[5]), int(tile[6])
            # the tile's keys [0, tsh) u [twl, tkh) lie in the pair's ranges
            if tsh > twl:   # merged ranges: [0, tkh)
                tsh, twl = 0, 0
            assert _inside(0, tsh, 0, sh) or _inside(0, tsh, wl_, kh), (rec, tile)
            assert _inside(twl, tkh, wl_, kh) or (sh == 0 and wl_ == 0 and tkh <= kh), (rec, tile)
        costs.append(_walk_tiles(segs, sh, wl_, kh))
        if skip:
            lo, hi = skip & 0xffff, skip >> 16
            assert 0 <= lo < hi <= len(segs), (rec, skip)
            for d, ln in segs[lo:hi]:
                assert d >= sh, "a skipped segment meets the sink range"
                assert d + ln <= wl_, "a skipped segment meets the window range"
            skipped_any = True
    assert real == plan.info["dense_tiles"], "every tile lies in exactly one pair"
    assert all(a >= b for a, b in zip(costs, costs[1:])), "pairs are ordered longest first"
    if name == "ctx16k":
        assert skipped_any, "Local pairs far from the sink skip segments"
    # the side kernel's share: the pairs of at most 8 key tiles at the end of
    # the list
    tail = 0
    for cst in reversed(costs):
        if cst > 8:
            break
        tail += 1
    assert plan.info["side_pairs"] == tail
    if name in ("ctx16k", "ctx128k_mini", "flash_mini", "ctx128k_vrope_mini"):
        assert tail > 0, "Local pairs are short"


def test_no_side_pairs_flag():
    """RK_PLAN_NO_SIDE_PAIRS keeps every pair on the 4-CTA clusters; the pair
    list itself does not change."""
    wl, plan = _host_plan("ctx16k")
    assert plan.info["side_pairs"] > 0
    bm, _ = build_bitmap(wl)
    flat, begins = segments_for_abi(wl)
    segs = [(0x10000000 + i * 0x1000000, s[1], s[2], s[3]) for i, s in enumerate(flat)]
    off = B.SegAttnPlan(segments=segs, seg_begin=begins,
                        q_row_begin=[r.q_row_begin for r in wl.requests], num_heads=wl.H,
                        d_nope=wl.d_nope, d_rope=wl.d_rope, rope_base=wl.rope_base,
                        softmax_scale=wl.scale, head_role=wl.head_role, sink=wl.sink,
                        window=wl.window, bitmap=bm,
                        flags=B.RK_PLAN_HOST_ONLY | B.RK_PLAN_NO_SIDE_PAIRS)
    assert off.info["side_pairs"] == 0
    assert np.array_equal(off.pairs(), plan.pairs())
