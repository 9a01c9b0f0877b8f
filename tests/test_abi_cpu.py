"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, rejects bad descriptors before touching the device, and its
host plan counts exactly the attended pairs the oracle's visibility rule
gives."""
import os
import re

import numpy as np
import pytest

import oracle as O
from position_independent_kv_gb300 import binding as B
from position_independent_kv_gb300 import build as BUILD
from position_independent_kv_gb300.protected import build_bitmap
from position_independent_kv_gb300.workloads import make_geometry

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    BUILD.build()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(rk_\w+)\s*\(", txt))
    return names


def test_exports_every_declared_symbol():
    L = B.lib()
    declared = _declared()
    assert declared >= set(B.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings():
    for code in range(12):
        assert B.status_string(code)
    assert B.status_string(0) == "ok"
    assert B.status_string(999) == "unknown status"


def _fake_addr(i, s):
    return 0x10000000 + i * 0x1000000


def _host_plan(name, **over):
    wl = make_geometry(name, 0)
    bm, _ = build_bitmap(wl)
    from position_independent_kv_gb300.workloads import segments_for_abi
    flat, begins = segments_for_abi(wl)
    segs = [(_fake_addr(i, s), s[1], s[2], s[3]) for i, s in enumerate(flat)]
    kw = dict(segments=segs, seg_begin=begins, q_row_begin=[r.q_row_begin for r in wl.requests],
              num_heads=wl.H, d_nope=wl.d_nope, d_rope=wl.d_rope, rope_base=wl.rope_base,
              softmax_scale=wl.scale, head_role=wl.head_role, sink=wl.sink, window=wl.window,
              bitmap=bm, flags=B.RK_PLAN_HOST_ONLY | (B.RK_PLAN_V_ROPE if wl.v_rope else 0))
    kw.update(over)
    return wl, B.SegAttnPlan(**kw)


def _expect(status, **over):
    with pytest.raises(B.RkError) as ei:
        _host_plan("tiny", **over)
    assert ei.value.status == status, str(ei.value)


def test_plan_errors():
    wl, plan = _host_plan("tiny")
    segs = plan._keep[0]
    _expect(2, num_heads=12)                  # not a multiple of 8
    _expect(5, d_nope=256)                    # dims not compiled
    _expect(2, rope_base=1.0)
    _expect(2, softmax_scale=0.0)
    _expect(2, window=-1)
    _expect(2, flags=B.RK_PLAN_HOST_ONLY | 128)
    _expect(2, q_row_begin=[576])             # beyond T
    _expect(2, head_role=np.array([0, 0, 0, 0, 0, 0, 0, 2], np.uint8))
    _expect(2, seg_begin=[0, 0])              # empty request
    # overlap: second segment starts inside the first
    bad = [segs[0], (segs[1][0], 256, 200, False), segs[2]]
    _expect(3, segments=bad)
    # gap: second segment leaves rows 256..299 uncovered
    bad = [segs[0], (segs[1][0], 256, 300, False), (segs[2][0], 64, 556, True)]
    _expect(4, segments=bad)
    # misaligned latent pointer
    bad = [(segs[0][0] + 8, 256, 0, False), segs[1], segs[2]]
    _expect(10, segments=bad)
    bad = [(0, 256, 0, False), segs[1], segs[2]]
    _expect(1, segments=bad)
    bad = [segs[0], (segs[1][0], 0, 256, False), segs[2]]
    _expect(2, segments=bad)


def test_host_only_plan_refuses_forward():
    _, plan = _host_plan("tiny")
    with pytest.raises(B.RkError) as ei:
        plan.forward(0x1000, 0x2000, 0x3000, stream=0)
    assert ei.value.status == 9
    with pytest.raises(B.RkError) as ei:
        plan.forward_host(0x4000, 0x5000, 0x6000, 0x1000, 0x2000, 0x3000, stream=0)
    assert ei.value.status == 9
    with pytest.raises(B.RkError) as ei:  # a missing host array is reported first
        plan.forward_host(0, 0x5000, 0x6000, 0x1000, 0x2000, 0x3000, stream=0)
    assert ei.value.status == 1


def test_lse_merge_argument_errors():
    L = B.lib()
    assert L.rk_lse_merge(None, None, 1, 1, 1, 1, None, None, None) == 1
    assert L.rk_lse_merge(16, 32, 0, 1, 1, 1, 64, 128, None) == 2
    assert L.rk_lse_merge(16, 32, 1, 1, 1, 4096, 64, 128, None) == 2
    assert L.rk_lse_merge(18, 32, 1, 1, 1, 8, 64, 128, None) == 10


@pytest.mark.parametrize("name", ["tiny", "flash_mini", "varlen_mini", "ctx128k_mini",
                                  "decode_mini", "tiny_wide", "flash", "decode",
                                  "flash_vrope_mini", "ctx128k_vrope_mini", "decode_vrope_mini"])
def test_plan_counts_attended_pairs(name):
    """The plan's pair accounting equals the oracle's visibility rule summed
    over the computed rows (Global heads) and the protected computed rows
    (Local heads)."""
    wl, plan = _host_plan(name)
    info = plan.info
    _, rows = build_bitmap(wl)
    HG = int(wl.head_role.sum())
    HL = wl.H - HG
    pg = pl = nprot = 0
    for req, prot in zip(wl.requests, rows):
        p = np.arange(req.q_row_begin, req.T)
        pg += HG * int((p + 1).sum())
        sel = p[prot[req.q_row_begin:]] if len(p) else p
        nprot += len(sel)
        if len(sel) < 5000:
            pl += HL * sum(len(O.visible_keys(int(x), False, wl.sink, wl.window)) for x in sel)
        else:
            lo = np.maximum(0, sel - wl.window)
            cnt = np.where(lo <= wl.sink, sel + 1, np.minimum(wl.sink, sel + 1) + sel - lo + 1)
            pl += HL * int(cnt.sum())
    assert info["rows"] == wl.rows
    assert info["pairs_global"] == pg
    assert info["pairs_local"] == pl
    assert info["protected_local_rows"] == nprot
    assert info["performed_pairs"] >= pg + pl
    assert info["num_global_heads"] == HG and info["num_local_heads"] == HL


@pytest.mark.parametrize("name", ["flash_mini", "varlen_mini", "ctx128k_mini", "flash", "ctx16k",
                                  "ctx128k"])
def test_pair_plan_work_bounds(name):
    """For d = (512, 64) the default plan pairs tcgen05 tiles on 4-CTA
    clusters (kernel 3), RK_PLAN_CTA_PAIR on CTA pairs (kernel 2), and
    RK_PLAN_SINGLE_CTA keeps one tile per two CTAs (kernel 1).  Pairing walks the union of two tiles' key ranges: the
    pairing rule bounds the extra key tiles by 1/8, and a merged range can
    also save a key tile where a tile's sink and window ranges split one
    128-key block.  Either way every attended pair is still covered."""
    _, pp = _host_plan(name)
    _, p2 = _host_plan(name, flags=B.RK_PLAN_HOST_ONLY | B.RK_PLAN_CTA_PAIR)
    _, ps = _host_plan(name, flags=B.RK_PLAN_HOST_ONLY | B.RK_PLAN_SINGLE_CTA)
    a, b = pp.info, ps.info
    assert a["kernel"] == 3 and p2.info["kernel"] == 2 and b["kernel"] == 1
    assert p2.info["performed_pairs"] == a["performed_pairs"]
    assert a["dense_tiles"] == b["dense_tiles"]
    assert a["performed_pairs"] <= b["performed_pairs"] * 9 // 8
    assert a["performed_pairs"] >= a["pairs_global"] + a["pairs_local"]


def test_vrope_plan_rules():
    """RK_PLAN_V_ROPE: the value is the whole latent row (d_v = d_k = 512 for
    d = (448, 64)); it runs on the 4-CTA kernel and the split decode kernel
    only, and needs exactly those dims."""
    V = B.RK_PLAN_HOST_ONLY | B.RK_PLAN_V_ROPE
    wl, plan = _host_plan("flash_vrope_mini", flags=V)
    info = plan.info
    assert info["kernel"] == 3 and info["d_v"] == 512 and info["d_nope"] == 448
    assert _host_plan("flash_mini")[1].info["d_v"] == 512
    assert _host_plan("tiny")[1].info["d_v"] == 128
    for name, flags in [("flash_mini", V),                          # (512, 64) with the flag
                        ("flash_vrope_mini", B.RK_PLAN_HOST_ONLY),  # (448, 64) without it
                        ("flash_vrope_mini", V | B.RK_PLAN_LEGACY_MMA),
                        ("flash_vrope_mini", V | B.RK_PLAN_SINGLE_CTA),
                        ("flash_vrope_mini", V | B.RK_PLAN_CTA_PAIR)]:
        with pytest.raises(B.RkError) as ei:
            _host_plan(name, flags=flags)
        assert ei.value.status == 5, (name, flags)
    # decode: same geometry as decode_mini; the partials are d_k wide
    _, pd = _host_plan("decode_vrope_mini", flags=V)
    _, pn = _host_plan("decode_mini")
    assert pd.info["split_chunks"] == pn.info["split_chunks"] > 0
    parts = pd.info["split_chunks"]
    body = ((parts * 8 * 512 * 4 + parts * 8 * 4 + 255) // 256) * 256
    # plus the 4-CTA kernel's work queues (its Local tiles): 8 launches' worth
    # of a claim counter and 64-entry rings for 40 clusters and 8 side pairs
    queue = 8 * (256 + (40 + 8) * 64 * 8)
    assert pd.info["kernel"] == 3
    assert body + queue < pd.workspace_bytes <= body + 256 + 4 * parts + queue


@pytest.mark.parametrize("name", ["edge_sink0_w0", "edge_tiny_decode", "edge_h8", "edge_many_segs"])
def test_edge_plans_count_attended_pairs(name):
    """The degenerate geometries plan with the exact attended-pair counts
    (H = 8 takes the mma.sync tiles, the others the 4-CTA kernel)."""
    test_plan_counts_attended_pairs(name)
    _, plan = _host_plan(name)
    assert plan.info["kernel"] == (0 if name == "edge_h8" else 3)


@pytest.mark.parametrize("name", ["tiny", "tiny_wide"])
def test_small_head_plans_take_the_tcgen05_tiles(name):
    """d = (128, 32) plans on the small-head tcgen05 kernel (4) by default and
    on the mma.sync tiles with RK_PLAN_LEGACY_MMA; both count the same
    attended pairs, the tcgen05 tiles 128 query pairs x 128 keys each."""
    wl, plan = _host_plan(name)
    _, legacy = _host_plan(name, flags=B.RK_PLAN_HOST_ONLY | B.RK_PLAN_LEGACY_MMA)
    assert plan.info["kernel"] == 4 and legacy.info["kernel"] == 0
    for k in ("pairs_global", "pairs_local", "protected_local_rows"):
        assert plan.info[k] == legacy.info[k]
    assert plan.info["performed_pairs"] % (128 * 128) == 0
    assert plan.info["performed_pairs"] >= plan.info["pairs_global"] + plan.info["pairs_local"]


def test_lse_merge_no_rows_is_a_no_op():
    L = B.lib()
    assert L.rk_lse_merge(16, 32, 3, 0, 4, 8, 64, 128, None) == 0
