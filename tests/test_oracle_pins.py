"""Pins for the CPU oracle: closed forms, library routines, brute force and
the pages' worked examples.  Each test names what a plausible mistake in the
oracle would break."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O


def _rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- RoPE ----

def test_rope_offset_identity():
    """R(-D) R(p) q . R(j) k == R(p) q . R(j + D) k  (RedKnot-MLA paper,
    RoPE-orthogonality paragraph; blog relocation equation).  Catches a sign
    error in the relocation direction or a non-additive rotation."""
    rng = _rng(1)
    for d in (32, 64):
        for _ in range(200):
            q = rng.standard_normal(d)
            k = rng.standard_normal(d)
            D = float(rng.integers(0, 2 ** 17))
            p = float(rng.integers(0, 2 ** 17))
            j = float(rng.integers(0, 2 ** 13))
            lhs = O.rotate(O.rotate(O.rotate(q, p, 1e4), -D, 1e4), 0.0, 1e4) @ O.rotate(k, j, 1e4)
            rhs = O.rotate(q, p, 1e4) @ O.rotate(k, j + D, 1e4)
            assert abs(lhs - rhs) <= 1e-9 * np.linalg.norm(q) * np.linalg.norm(k)


def test_rope_closed_forms():
    """Orthogonality (norm kept), theta_0 = 1 (pair 0 turns by exactly p
    radians: R(pi) = -1 on that pair), the last pair's frequency
    base^(-(d-2)/d), and R(a) R(b) = R(a + b)."""
    rng = _rng(2)
    x = rng.standard_normal(64)
    for p in (0.0, 1.0, 77.0, 131071.0):
        assert np.isclose(np.linalg.norm(O.rotate(x, p, 1e4)), np.linalg.norm(x), rtol=1e-13)
    e0 = np.zeros(64)
    e0[0] = 1.0
    r = O.rotate(e0, math.pi, 1e4)
    assert np.allclose(r[:2], [-1.0, 0.0], atol=1e-15) and np.allclose(r[2:], 0.0)
    th = O.rope_theta(64, 1e4)
    assert th[0] == 1.0
    assert np.isclose(th[-1], 1e4 ** (-62 / 64), rtol=1e-15)
    # pair 31 turns by theta_31 * p: after p = 2 pi / theta_31 it is back
    e31 = np.zeros(64)
    e31[62] = 1.0
    back = O.rotate(e31, 2 * math.pi / th[-1], 1e4)
    assert np.allclose(back, e31, atol=1e-9)
    a, b = 1234.0, -567.0
    assert np.allclose(O.rotate(O.rotate(x, a, 1e4), b, 1e4), O.rotate(x, a + b, 1e4), atol=1e-10)


# -------------------------------------------------------------- merge -----

def test_lse_merge_equals_unsegmented():
    """Segmented statistics merged by log-sum-exp equal attention over the
    whole key set (paper, RoPE-orthogonality paragraph).  Also checks lse
    against scipy's logsumexp.  Catches a dropped weight or a wrong sign in
    the rescale."""
    from scipy.special import logsumexp
    rng = _rng(3)
    for trial in range(30):
        n = int(rng.integers(1, 300))
        h, dk, dv = 4, 24, 16
        q = rng.standard_normal((h, dk))
        K = rng.standard_normal((n, dk)) * 2
        V = rng.standard_normal((n, dv))
        full_o, full_l = O.attend(q, K, V[:, :dv], 0.3)
        assert np.allclose(full_l, logsumexp(0.3 * q @ K.T, axis=1), atol=1e-12)
        cuts = np.sort(rng.integers(0, n + 1, size=int(rng.integers(0, 6))))
        edges = [0, *cuts.tolist(), n]
        parts = [O.attend_partial(q, K[a:b], V[a:b], 0.3) for a, b in zip(edges[:-1], edges[1:])]
        mo, ml = O.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        assert np.allclose(mo, full_o, atol=1e-12)
        assert np.allclose(ml, full_l, atol=1e-12)


def test_lse_merge_all_empty():
    o, l = O.lse_merge(np.zeros((3, 2, 5)), np.full((3, 2), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(l))


# ------------------------------------------------------------ masks -------

def test_window_worked_example(golden_dir):
    """Blog 'Insight 1' worked example: w = 256, token 1000 sees 744..1000
    plus the sink."""
    g = json.load(open(os.path.join(golden_dir, "window_worked_example.json")))
    keys = O.visible_keys(g["row"], False, g["sink"], g["window"])
    expect = list(range(g["sink"])) + list(range(g["window_first"], g["window_last"] + 1))
    assert keys.tolist() == expect
    assert len(keys) == g["sink"] + g["window"] + 1
    assert O.visible_keys(g["row"], True, g["sink"], g["window"]).tolist() == list(range(g["row"] + 1))


def test_visible_keys_edges():
    # window reaching into the sink: no duplicates, contiguous
    assert O.visible_keys(10, False, 4, 8).tolist() == list(range(11))
    assert O.visible_keys(13, False, 4, 8).tolist() == [0, 1, 2, 3] + list(range(5, 14))
    assert O.visible_keys(2, False, 4, 8).tolist() == [0, 1, 2]
    assert O.visible_keys(0, False, 4, 0).tolist() == [0]


def test_head_role_ceiling(golden_dir):
    """Profiles paragraph: one Global head per group of eight; ceilings
    75.29 % (Flash 3F-37R-3F, 56/64) and 78.89 % (Pro 3F-55R-3F, 112/128)."""
    from position_independent_kv_gb300.workloads import SPECS, _roles
    g = json.load(open(os.path.join(golden_dir, "head_row_ceiling.json")))
    for prof in g["profiles"].values():
        layers = prof["fence_first"] + prof["reusable"] + prof["fence_last"]
        ceil = prof["reusable"] / layers * prof["local"] / prof["heads"]
        assert round(100 * ceil, 2) == prof["ceiling_pct"]
        role = _roles(prof["heads"])
        assert int((role == 0).sum()) == prof["local"]
        assert all(role[8 * i:8 * i + 8].sum() == 1 for i in range(prof["heads"] // 8))
    assert SPECS["flash"].H == 64 and SPECS["ctx128k"].H == 128


# ------------------------------------------------------- brute force ------

def _tiny_case(rng, T_cached_parts, n_new, H=2, d_nope=4, d_rope=4):
    d_k = d_nope + d_rope
    lens = list(T_cached_parts) + [n_new]
    order = rng.permutation(len(T_cached_parts))
    deltas = [0] * len(lens)
    pos = 0
    for j in order:
        deltas[j] = pos
        pos += lens[j]
    deltas[-1] = pos
    T = pos + n_new
    segs = []
    for j, n in enumerate(lens):
        segs.append((rng.standard_normal((n, d_k)), deltas[j], j == len(lens) - 1))
    role = np.array([0, 1] * (H // 2), dtype=np.uint8)
    return segs, T, role, d_nope


def test_brute_force_matches_vectorised():
    """A pure-Python triple loop (no NumPy arithmetic) against the vectorised
    oracle on tiny shapes: catches index, transpose, mask and assembly
    mistakes."""
    rng = _rng(4)
    for trial in range(12):
        parts = [int(x) for x in rng.integers(1, 9, size=int(rng.integers(1, 4)))]
        n_new = int(rng.integers(1, 6))
        segs, T, role, d_nope = _tiny_case(rng, parts, n_new)
        H, d_k = len(role), segs[0][0].shape[1]
        qb = int(rng.integers(0, T)) if trial % 3 == 0 else 0
        q = rng.standard_normal((T - qb, H, d_k)) * 1.5
        prot = rng.random(T) < 0.4
        oin = rng.standard_normal((T - qb, H, d_nope))
        lin = rng.standard_normal((T - qb, H))
        sink, window = int(rng.integers(0, 3)), int(rng.integers(0, 6))
        base = 10000.0 if trial % 2 else 100.0
        scale = 0.7
        Ov, Lv = O.seg_attn_request(q, segs, T, qb, role, d_nope, base, scale, sink, window,
                                    prot, oin, lin)
        Ob, Lb = O.brute_force(q.tolist(), [(s[0].tolist(), s[1], s[2]) for s in segs], T, qb,
                               role.tolist(), d_nope, base, scale, sink, window, prot.tolist(),
                               oin.tolist(), lin.tolist())
        assert np.allclose(Ov, np.array(Ob), atol=1e-12)
        assert np.allclose(Lv, np.array(Lb), atol=1e-12)


# -------------------------------------------------- special cases ---------

def _absolute_frame_case(rng, lens, n_new, H, d_nope, d_rope, base, q_scale=3.0):
    """Keys drawn directly at absolute positions; canonical latents obtained
    by turning each segment back by its offset.  The oracle must turn them
    forward again."""
    d_k = d_nope + d_rope
    T = sum(lens) + n_new
    K_abs = rng.standard_normal((T, d_k))
    order = rng.permutation(len(lens))
    deltas = [0] * len(lens)
    pos = 0
    for j in order:
        deltas[j] = pos
        pos += lens[j]
    segs = []
    for j, n in enumerate(list(lens) + [n_new]):
        d = deltas[j] if j < len(lens) else pos
        lat = K_abs[d:d + n].copy()
        lat[:, d_nope:] = O.rotate(lat[:, d_nope:], -float(d), base)
        segs.append((lat, d, j == len(lens)))
    q = rng.standard_normal((T, H, d_k)) * q_scale / math.sqrt(d_k)
    return segs, T, K_abs, q


def test_global_equals_causal_sdpa():
    """All-Global heads reduce to textbook causal softmax attention on the
    keys at their absolute positions: torch's scaled_dot_product_attention
    (fp64, is_causal) and torch.logsumexp.  Catches a relocation sign error,
    a causal off-by-one and a wrong scale."""
    rng = _rng(5)
    H, d_nope, d_rope = 3, 16, 8
    segs, T, K_abs, q = _absolute_frame_case(rng, [13, 29, 7], 11, H, d_nope, d_rope, 1e4)
    role = np.ones(H, np.uint8)
    scale = 1 / math.sqrt(d_nope + d_rope)
    Ov, Lv = O.seg_attn_request(q, segs, T, 0, role, d_nope, 1e4, scale, 4, 5,
                                np.zeros(T, bool), np.zeros((T, H, d_nope)), np.zeros((T, H)))
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(K_abs)[None].expand(H, T, -1)
    vt = torch.from_numpy(K_abs[:, :d_nope])[None].expand(H, T, -1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    assert np.allclose(Ov, ref.permute(1, 0, 2).numpy(), atol=1e-12)
    sc = scale * torch.einsum("htd,sd->hts", qt, torch.from_numpy(K_abs))
    sc = sc.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), 1), float("-inf"))
    assert np.allclose(Lv, torch.logsumexp(sc, -1).T.numpy(), atol=1e-12)


def test_local_all_protected_equals_masked_sdpa():
    """Eq. (4) exactness reading: with every row protected the Local output
    is dense sink+window attention on every row (paper, sentence after eq.
    (4)); checked against SDPA with an explicit boolean mask built from the
    pinned visibility rule."""
    rng = _rng(6)
    H, d_nope, d_rope = 4, 16, 8
    segs, T, K_abs, q = _absolute_frame_case(rng, [20, 9, 31], 6, H, d_nope, d_rope, 1e4)
    role = np.zeros(H, np.uint8)
    sink, window = 3, 7
    scale = 0.31
    Ov, Lv = O.seg_attn_request(q, segs, T, 0, role, d_nope, 1e4, scale, sink, window,
                                np.ones(T, bool), np.zeros((T, H, d_nope)), np.zeros((T, H)))
    mask = torch.zeros(T, T, dtype=torch.bool)
    for p in range(T):
        mask[p, torch.from_numpy(O.visible_keys(p, False, sink, window))] = True
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(K_abs)[None].expand(H, T, -1)
    vt = torch.from_numpy(K_abs[:, :d_nope])[None].expand(H, T, -1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    assert np.allclose(Ov, ref.permute(1, 0, 2).numpy(), atol=1e-12)


def test_wide_window_local_equals_global():
    """A Local window covering the whole context equals Global."""
    rng = _rng(7)
    H = 4
    segs, T, _, q = _absolute_frame_case(rng, [17, 23], 9, H, 8, 8, 1e4)
    args = (q, segs, T, 0)
    rest = (8, 1e4, 0.4, 2, T + 5, np.ones(T, bool), np.zeros((T, H, 8)), np.zeros((T, H)))
    Og, Lg = O.seg_attn_request(*args, np.ones(H, np.uint8), *rest)
    Ol, Ll = O.seg_attn_request(*args, np.zeros(H, np.uint8), *rest)
    assert np.allclose(Og, Ol, atol=1e-13) and np.allclose(Lg, Ll, atol=1e-13)


def test_replacement_never_adds():
    """Unprotected Local rows keep the cached bytes exactly; protected rows do
    not depend on the cached values (paper: replaced, never double counted)."""
    rng = _rng(8)
    H = 4
    segs, T, _, q = _absolute_frame_case(rng, [15, 12], 5, H, 8, 8, 1e4)
    role = np.array([0, 0, 0, 1], np.uint8)
    prot = rng.random(T) < 0.5
    o1 = rng.standard_normal((T, H, 8))
    o2 = rng.standard_normal((T, H, 8))
    l1 = rng.standard_normal((T, H))
    A, LA = O.seg_attn_request(q, segs, T, 0, role, 8, 1e4, 0.4, 2, 3, prot, o1, l1)
    B, LB = O.seg_attn_request(q, segs, T, 0, role, 8, 1e4, 0.4, 2, 3, prot, o2, l1 + 1)
    new = np.zeros(T, bool)
    new[T - 5:] = True
    eff = prot | new
    for p in range(T):
        for h in range(3):
            if eff[p]:
                assert np.array_equal(A[p, h], B[p, h]) and LA[p, h] == LB[p, h]
            else:
                assert np.array_equal(A[p, h], o1[p, h]) and LA[p, h] == l1[p, h]
    assert np.array_equal(A[:, 3], B[:, 3])


def test_segment_order_invariance():
    rng = _rng(9)
    H = 2
    segs, T, _, q = _absolute_frame_case(rng, [11, 5, 8], 4, H, 8, 8, 1e4)
    rest = (np.array([0, 1], np.uint8), 8, 1e4, 0.5, 1, 3, np.ones(T, bool),
            np.zeros((T, H, 8)), np.zeros((T, H)))
    A, LA = O.seg_attn_request(q, segs, T, 0, *rest)
    B, LB = O.seg_attn_request(q, segs[::-1], T, 0, *rest)
    assert np.array_equal(A, B) and np.array_equal(LA, LB)


def test_decode_rows_subset():
    """Evaluating only the last row (decode) equals the last row of the full
    evaluation."""
    rng = _rng(10)
    H = 4
    segs, T, _, q = _absolute_frame_case(rng, [9, 14], 1, H, 8, 8, 1e4)
    role = np.array([0, 1, 0, 1], np.uint8)
    args = (segs, T)
    full = O.seg_attn_request(q, *args, 0, role, 8, 1e4, 0.5, 2, 4, np.zeros(T, bool),
                              np.zeros((T, H, 8)), np.zeros((T, H)))
    last = O.seg_attn_request(q[T - 1:], *args, T - 1, role, 8, 1e4, 0.5, 2, 4,
                              np.zeros(T, bool), np.zeros((1, H, 8)), np.zeros((1, H)))
    assert np.allclose(full[0][-1], last[0][0], atol=1e-14)
    assert np.allclose(full[1][-1], last[1][0], atol=1e-14)
