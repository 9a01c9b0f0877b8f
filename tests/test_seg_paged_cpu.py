"""SegPagedAttention C ABI without a GPU: host-only plans count exactly the
attended pairs of the oracle's visibility rule, visit only the sink and
window pages of Local heads, and refuse bad descriptors before any launch."""
import numpy as np
import pytest

import oracle as O
from position_independent_kv_gb300 import binding as B
from position_independent_kv_gb300 import build as BUILD
from position_independent_kv_gb300.paged_workloads import PAGE, make_paged_geometry


@pytest.fixture(scope="module", autouse=True)
def built():
    BUILD.build()


def _plan(pw, flags=0, **over):
    kw = dict(seq_len=pw.seq_len, q_row_begin=pw.q_row_begin, num_q_heads=pw.Hq,
              num_kv_heads=pw.Hkv, block_table=pw.block_table, num_pages=pw.num_pages,
              kv_role=pw.kv_role, sink=pw.sink, window=pw.window, softmax_scale=pw.scale,
              flags=B.RK_SEGPAGED_HOST_ONLY | flags)
    kw.update(over)
    return B.SegPagedPlan(**kw)


@pytest.mark.parametrize("name", ["paged_mini", "paged_mini_g4", "paged_mini_g1",
                                  "paged_mini_g16", "paged_decode_mini", "paged_decode_long_mini",
                                  "paged_decode_g16_long", "paged_decode_g1_long", "paged_decode_g4", "paged_tail_g1",
                                  "paged_tail_g2", "paged_tail_g4_split",
                                  "qwen32b_16k"])
def test_pair_counts_and_blocks(name):
    pw = make_paged_geometry(name, 0)
    info = _plan(pw).info
    G = pw.G
    pairs = 0
    for T, qb in zip(pw.seq_len, pw.q_row_begin):
        p = np.arange(qb, T)
        for g in range(pw.Hkv):
            if pw.kv_role[g]:
                pairs += G * int((p + 1).sum())
            elif len(p) < 3000:
                pairs += G * sum(len(O.visible_keys(int(x), False, pw.sink, pw.window)) for x in p)
            else:
                lo = np.maximum(0, p - pw.window)
                cnt = np.where(lo <= pw.sink, p + 1, np.minimum(pw.sink, p + 1) + p - lo + 1)
                pairs += G * int(cnt.sum())
    assert info["pairs"] == pairs and info["rows"] == pw.rows and info["group"] == G
    # 16, 128 or 256 query pairs per issued block (decode, one or two sub-tiles)
    assert info["kv_blocks"] * 16 * PAGE <= info["performed_pairs"] <= info["kv_blocks"] * 256 * PAGE
    assert info["performed_pairs"] >= pairs
    # the dense + mask arm walks every block up to each tile's last row
    if not (pw.block_table < 0).any():
        dense = _plan(pw, B.RK_SEGPAGED_DENSE_MASK).info
        assert dense["pairs"] == pairs and dense["kv_blocks"] >= info["kv_blocks"]


def test_qwen_128k_work():
    """The 128K prefill: Local tiles read at most a few pages, Global tiles
    up to the whole prompt; dense + mask reads every block for every head."""
    pw = make_paged_geometry("qwen32b_128k", 0)
    a = _plan(pw).info
    d = _plan(pw, B.RK_SEGPAGED_DENSE_MASK).info
    assert a["tiles"] == 8 * 131072 // 32
    assert d["kv_blocks"] > 7 * a["kv_blocks"] // 2
    assert a["pairs"] == d["pairs"]


def test_plan_errors():
    pw = make_paged_geometry("paged_mini", 0)

    def expect(status, **over):
        flags = over.pop("flags", 0)
        with pytest.raises(B.RkError) as ei:
            _plan(pw, flags, **over)
        assert ei.value.status == status, str(ei.value)

    expect(2, num_q_heads=15)                       # not a multiple of Hkv
    expect(5, num_q_heads=6, num_kv_heads=2)        # G = 3
    expect(5, head_dim=64)
    expect(5, page_size=64)
    expect(2, q_row_begin=np.array([1000, 0]))      # beyond T
    expect(2, sink=-1)
    expect(2, flags=8)
    expect(2, kv_role=np.array([0, 2], np.uint8))
    bad = pw.block_table.copy()
    bad[0, 0, 3] = -1                               # a needed page is missing
    expect(2, block_table=bad)
    bad = pw.block_table.copy()
    bad[1, 1, 0] = pw.num_pages                     # page out of range
    expect(2, block_table=bad)
    # a decode geometry whose Local heads dropped pages cannot run dense + mask
    pd = make_paged_geometry("paged_decode_mini", 0)
    assert (pd.block_table < 0).any()
    _plan(pd)
    with pytest.raises(B.RkError) as ei:
        _plan(pd, B.RK_SEGPAGED_DENSE_MASK)
    assert ei.value.status == 2


def test_host_only_refuses_forward():
    pw = make_paged_geometry("paged_mini", 0)
    plan = _plan(pw)
    with pytest.raises(B.RkError) as ei:
        plan.forward(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, None, stream=0)
    assert ei.value.status == 9


def test_decode_split_parts_and_workspace():
    """Decode rows (at most 16 query pairs) of Global heads with long walks
    (more than 48 blocks) are split into parts of 32 blocks; the workspace
    holds one fp32 partial and one LSE per used pair of every part, plus a
    ticket per split tile."""
    pw = make_paged_geometry("paged_decode_long_mini", 0)
    plan = _plan(pw)
    info = plan.info
    parts = 0
    lanes = 0
    split = 0
    for T in pw.seq_len:
        nb = (int(T) + PAGE - 1) // PAGE
        for g in range(pw.Hkv):
            if pw.kv_role[g] and nb > 48:
                np_ = (nb + 31) // 32
                parts += np_
                lanes += np_ * pw.G
                split += 1
    assert info["split_parts"] == parts
    want = ((lanes * 129 * 4 + 255) // 256) * 256 + split * 4
    assert split > 0 and plan.workspace_bytes == ((want + 255) // 256) * 256
    pq = make_paged_geometry("qwen32b_decode", 0)
    qi = _plan(pq).info
    assert qi["split_parts"] > 64 and qi["tiles"] > qi["split_parts"]


@pytest.mark.parametrize("name", ["paged_reloc_mini", "paged_reloc_g8", "paged_reloc_decode",
                                  "qwen32b_reloc_128k"])
def test_relocated_plans_use_single_sub_tiles(name):
    """With document offsets every tile is one sub-tile of 128 / G rows on the
    one-sub-tile kernel: 128 query pairs per issued block, the same attended
    pairs and blocks as the plan without offsets."""
    pw = make_paged_geometry(name, 0)
    rel = _plan(pw, block_delta=pw.block_delta, rope_base=pw.rope_base).info
    plain = _plan(pw).info
    assert rel["pairs"] == plain["pairs"] and rel["rows"] == plain["rows"]
    assert rel["performed_pairs"] == rel["kv_blocks"] * 128 * PAGE
    rows_per = 128 // pw.G
    want_tiles = 0
    for T, qb in zip(pw.seq_len, pw.q_row_begin):
        want_tiles += pw.Hkv * ((int(T) - int(qb) + rows_per - 1) // rows_per)
    assert rel["tiles"] >= want_tiles     # split parts add tiles, never remove them


def test_relocated_plan_errors():
    pw = make_paged_geometry("paged_reloc_mini", 0)
    bad = pw.block_delta.copy()
    bad[0, 1] = 1 << 40                            # offset beyond int32
    with pytest.raises(B.RkError) as ei:
        _plan(pw, block_delta=bad)
    assert ei.value.status == 2
    with pytest.raises(B.RkError) as ei:
        _plan(pw, block_delta=pw.block_delta, rope_base=0.5)
    assert ei.value.status == 2
