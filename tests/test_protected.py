"""The host protected-row builder against the oracle's independent one, bit
for bit, plus the properties the rule fixes."""
import numpy as np
import pytest

import oracle as O
from position_independent_kv_gb300 import protected as P
from position_independent_kv_gb300.workloads import SPECS, make_geometry

NAMES = ["tiny", "flash", "varlen", "ctx128k", "decode", "flash_mini", "varlen_mini",
         "ctx128k_mini", "decode_mini"]


@pytest.mark.parametrize("name", NAMES)
def test_bitmap_matches_oracle(name):
    wl = make_geometry(name, 0)
    words, rows = P.build_bitmap(wl)
    off = 0
    r = wl.rule
    for req, prot in zip(wl.requests, rows):
        segs = [(s.n, s.delta, s.is_new) for s in req.segments]
        ref = O.build_protected(req.T, segs, r.boundary, r.p_random, r.budget, r.none,
                                req.u, req.perm)
        assert np.array_equal(prot, ref)
        nw = (req.T + 31) // 32
        assert np.array_equal(words[off:off + nw], O.bitmap_words(ref))
        off += nw
    assert off == len(words)


def test_tiny_protected_rows():
    """Tiny workload: the 64 query rows plus the first/last 16 rows of each
    of the two 256-row segments."""
    wl = make_geometry("tiny", 0)
    _, rows = P.build_bitmap(wl)
    prot = rows[0]
    expect = set(range(512, 576)) | set(range(0, 16)) | set(range(240, 272)) | set(range(496, 512))
    assert set(np.nonzero(prot)[0].tolist()) == expect


@pytest.mark.parametrize("name,pct", [("varlen", 20), ("ctx128k", 25)])
def test_budget_count(name, pct):
    wl = make_geometry(name, 0)
    _, rows = P.build_bitmap(wl)
    req = wl.requests[0]
    new = np.zeros(req.T, bool)
    for s in req.segments:
        if s.is_new:
            new[s.delta:s.delta + s.n] = True
    C = int((~new).sum())
    cached_prot = int((rows[0] & ~new).sum())
    assert cached_prot == -(-pct * C // 100)
    assert rows[0][new].all()


def test_ctx128k_geometry():
    wl = make_geometry("ctx128k", 0)
    req = wl.requests[0]
    assert req.T == 131072 and len(req.segments) == 49
    new = [s for s in req.segments if s.is_new][0]
    assert new.delta == 98304 and new.n == 32768
    assert sorted(s.delta for s in req.segments if not s.is_new) == list(range(0, 98304, 2048))


def test_decode_geometry():
    wl = make_geometry("decode", 0)
    assert len(wl.requests) == 64
    for req in wl.requests:
        cached = [s for s in req.segments if not s.is_new]
        assert 4 <= len(cached) <= 32
        L = sum(s.n for s in cached)
        assert 8192 <= L <= 65536 and req.q_row_begin == L and req.T == L + 1
        spans = sorted((s.delta, s.n) for s in req.segments)
        pos = 0
        for d, n in spans:
            assert d == pos and n >= 1
            pos += n


def test_dirty_rows_protected_outside_the_budget():
    """The paper's D (dirty rows) joins the protected union; the budget fill
    (boundary first, then the permutation) is the same with or without it."""
    wl = make_geometry("varlen_mini", 0)
    r = wl.rule
    req = wl.requests[0]
    segs = [(s.n, s.delta, s.is_new) for s in req.segments]
    base = O.build_protected(req.T, segs, r.boundary, r.p_random, r.budget, r.none,
                             req.u, req.perm)
    rng = np.random.default_rng(3)
    dirty = rng.random(req.T) < 0.05
    got = O.build_protected(req.T, segs, r.boundary, r.p_random, r.budget, r.none,
                            req.u, req.perm, dirty=dirty)
    assert np.array_equal(got, base | dirty)
