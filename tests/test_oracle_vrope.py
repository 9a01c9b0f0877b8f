"""Pins of the oracle's output-phase restore (RedKnot-MLA paper: inverse
output RoPE R^-1 in the head-partition paragraph; "restores the output phase"
in the RoPE-orthogonality paragraph).  With the value equal to the packed
latent row, the output's rope slice is sum_k P_k R(k - p) v_k.  Each pin
fixes that from something other than the oracle's own code: brute force,
a one-hot attention whose output is a known latent row, and the per-segment
restore + merge order the kernels use."""
import math

import numpy as np

import oracle as O


def _rng(seed):
    return np.random.default_rng(seed)


def _case(rng, lens, n_new, H, d_nope, d_rope):
    """Canonical latents of shuffled contiguous segments plus new rows."""
    d_k = d_nope + d_rope
    order = rng.permutation(len(lens))
    deltas = [0] * len(lens)
    pos = 0
    for j in order:
        deltas[j] = pos
        pos += lens[j]
    segs = [(rng.standard_normal((n, d_k)), deltas[j], False) for j, n in enumerate(lens)]
    segs.append((rng.standard_normal((n_new, d_k)), pos, True))
    return segs, pos + n_new


def test_vrope_brute_force():
    """Pure-Python loops (value = relocated key row, output rope slice turned
    by R(-p)) against the vectorised oracle."""
    rng = _rng(21)
    for trial in range(8):
        H, d_nope, d_rope = 2, 4, 4
        lens = [int(x) for x in rng.integers(1, 8, size=int(rng.integers(1, 4)))]
        segs, T = _case(rng, lens, int(rng.integers(1, 5)), H, d_nope, d_rope)
        d_k = d_nope + d_rope
        role = np.array([0, 1], np.uint8)
        qb = int(rng.integers(0, T)) if trial % 2 else 0
        q = rng.standard_normal((T - qb, H, d_k))
        prot = rng.random(T) < 0.5
        oin = rng.standard_normal((T - qb, H, d_k))
        lin = rng.standard_normal((T - qb, H))
        base = 100.0 if trial % 2 else 10000.0
        Ov, Lv = O.seg_attn_request(q, segs, T, qb, role, d_nope, base, 0.6, 1, 3, prot, oin,
                                    lin, v_rope=True)
        Ob, Lb = O.brute_force(q.tolist(), [(s[0].tolist(), s[1], s[2]) for s in segs], T, qb,
                               role.tolist(), d_nope, base, 0.6, 1, 3, prot.tolist(),
                               oin.tolist(), lin.tolist(), v_rope=True)
        assert np.allclose(Ov, np.array(Ob), atol=1e-12)
        assert np.allclose(Lv, np.array(Lb), atol=1e-12)


def _one_hot_query(K_rel, k_star, d_nope, d_k, gap=400.0):
    """A query whose nope part points at key k_star so hard that every other
    visible key is at least `gap` nats below it (checked), rope part 0."""
    q = np.zeros(d_k)
    q[:d_nope] = K_rel[k_star, :d_nope]
    return q * (gap / np.dot(K_rel[k_star, :d_nope], K_rel[k_star, :d_nope]))


def test_vrope_diagonal_sees_canonical_row():
    """The first row of a segment, attending only to itself, returns that
    segment's canonical latent row 0 unchanged, rope slice included: its
    key sits at p = delta, so the relocation R(delta) and the inverse output
    RoPE R(-p) cancel exactly.  No rotation enters the expected value."""
    rng = _rng(22)
    d_nope, d_rope, H = 16, 8, 1
    d_k = d_nope + d_rope
    segs, T = _case(rng, [9, 13, 6], 3, H, d_nope, d_rope)
    for lat, delta, _ in segs:
        p = delta
        K, _ = O.relocate([(s[0], s[1]) for s in segs], T, d_nope, 1e4)
        q = np.zeros((1, H, d_k))
        q[0, 0] = _one_hot_query(K, p, d_nope, d_k)
        scores = K[:p + 1, :d_nope] @ q[0, 0, :d_nope]
        assert p == 0 or np.sort(scores)[-2] < scores[p] - 100.0
        o, _ = O.seg_attn_request(q, segs, T, p, np.ones(H, np.uint8), d_nope, 1e4, 1.0, 0, 0,
                                  np.zeros(T, bool), np.zeros((1, H, d_k)), np.zeros((1, H)),
                                  rows=[p], sampled=True, v_rope=True)
        assert np.allclose(o[0, 0], lat[0], atol=1e-12)


def test_vrope_one_hot_earlier_key():
    """Row p attending (one-hot) to key k* = delta* + j* of another segment
    returns [c_nope(j*) | R(delta* - p) k_rope(j*)]: the key's canonical rope
    slice moved by its own offset and back by the query's position."""
    rng = _rng(23)
    d_nope, d_rope, H = 16, 8, 2
    d_k = d_nope + d_rope
    base = 1e4
    segs, T = _case(rng, [11, 7, 15], 4, H, d_nope, d_rope)
    K, _ = O.relocate([(s[0], s[1]) for s in segs], T, d_nope, base)
    for lat, delta, is_new in segs:
        if is_new:
            continue
        j = int(rng.integers(0, lat.shape[0]))
        k_star = delta + j
        p = T - 1
        q = np.zeros((1, H, d_k))
        q[0, :] = _one_hot_query(K, k_star, d_nope, d_k)
        scores = K[:p + 1, :d_nope] @ q[0, 0, :d_nope]
        assert np.sort(scores)[-2] < scores[k_star] - 100.0
        o, _ = O.seg_attn_request(q, segs, T, p, np.ones(H, np.uint8), d_nope, base, 1.0, 0, 0,
                                  np.zeros(T, bool), np.zeros((1, H, d_k)), np.zeros((1, H)),
                                  rows=[p], sampled=True, v_rope=True)
        want = np.concatenate([lat[j, :d_nope], O.rotate(lat[j, d_nope:], float(delta - p), base)])
        assert np.allclose(o[0, 0], want, atol=1e-12)
        assert np.allclose(o[0, 1], want, atol=1e-12)


def test_vrope_segment_partials_restore_then_merge():
    """The kernels' order: per segment, attend the CANONICAL latent with the
    query's rope turned by R(-delta_i) (values unrotated), restore the
    partial's rope slice by R(+delta_i), merge the partials by log-sum-exp,
    then apply R(-p).  Equals the oracle's direct result (linearity of the
    rotation; the merge weights are scalars)."""
    rng = _rng(24)
    d_nope, d_rope, H = 8, 8, 3
    d_k = d_nope + d_rope
    base = 1e4
    segs, T = _case(rng, [10, 4, 12, 7], 5, H, d_nope, d_rope)
    q = rng.standard_normal((T, H, d_k)) * 2.0
    scale = 1 / math.sqrt(d_k)
    direct, dl = O.seg_attn_request(q, segs, T, 0, np.ones(H, np.uint8), d_nope, base, scale, 0,
                                    0, np.zeros(T, bool), np.zeros((T, H, d_k)),
                                    np.zeros((T, H)), v_rope=True)
    for p in (0, T // 3, T - 1):
        parts_o, parts_l = [], []
        for lat, delta, _ in segs:
            n = min(lat.shape[0], p + 1 - delta)
            qh = q[p].copy()
            qh[:, d_nope:] = O.rotate(qh[:, d_nope:], -float(delta), base)
            o, l = O.attend_partial(qh, lat[:max(n, 0)], lat[:max(n, 0)], scale)
            if n > 0:
                o[:, d_nope:] = O.rotate(o[:, d_nope:], float(delta), base)
            parts_o.append(o)
            parts_l.append(l)
        om, lm = O.lse_merge(np.array(parts_o), np.array(parts_l))
        om[:, d_nope:] = O.rotate(om[:, d_nope:], -float(p), base)
        assert np.allclose(om, direct[p], atol=1e-12)
        assert np.allclose(lm, dl[p], atol=1e-12)


def test_vrope_off_keeps_value_nope_only():
    """Without the flag the value is c_nope alone (the configs' reading); the
    nope columns of the two results coincide."""
    rng = _rng(25)
    d_nope, d_rope, H = 8, 8, 2
    segs, T = _case(rng, [6, 9], 3, H, d_nope, d_rope)
    q = rng.standard_normal((T, H, d_nope + d_rope))
    args = (q, segs, T, 0, np.array([1, 0], np.uint8), d_nope, 1e4, 0.5, 1, 2, np.ones(T, bool))
    a, la = O.seg_attn_request(*args, np.zeros((T, H, d_nope)), np.zeros((T, H)))
    b, lb = O.seg_attn_request(*args, np.zeros((T, H, d_nope + d_rope)), np.zeros((T, H)),
                               v_rope=True)
    assert a.shape[-1] == d_nope and b.shape[-1] == d_nope + d_rope
    assert np.allclose(a, b[..., :d_nope], atol=1e-13) and np.allclose(la, lb, atol=1e-13)
