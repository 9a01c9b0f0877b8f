"""Pins of the SegPagedAttention oracle (RedKnot blog, "Insight 3": per-head
pages, Global heads over the whole prompt, Local heads over sink + window,
no mask; same results as dense + mask).  Each pin fixes the oracle from
something other than its own code: pure-Python loops over the pages, torch's
scaled_dot_product_attention with GQA key/value repetition, page-layout
invariances and the dropped-pages claim."""
import math

import numpy as np
import pytest
import torch

import oracle as O


def _case(rng, T, Hq, Hkv, d, page_size, roles, drop_local=False, sink=2, window=5):
    """Logical K/V per KV head, scattered into shuffled physical pages."""
    nb = (T + page_size - 1) // page_size
    K = rng.standard_normal((Hkv, T, d))
    V = rng.standard_normal((Hkv, T, d))
    npages = Hkv * nb
    perm = rng.permutation(npages)
    kp = np.zeros((npages, page_size, d))
    vp = np.zeros((npages, page_size, d))
    table = np.full((Hkv, nb + 2), -1, dtype=np.int64)
    for g in range(Hkv):
        for b in range(nb):
            pg = int(perm[g * nb + b])
            n = min(page_size, T - b * page_size)
            kp[pg, :n] = K[g, b * page_size:b * page_size + n]
            vp[pg, :n] = V[g, b * page_size:b * page_size + n]
            table[g, b] = pg
    return K, V, kp, vp, table


def test_brute_force_over_pages():
    rng = np.random.default_rng(31)
    for trial in range(6):
        T, Hq, Hkv, d, ps = int(rng.integers(5, 19)), 4, 2, 4, int(rng.integers(2, 5))
        roles = np.array([trial % 2, 1 - trial % 2], np.uint8)
        K, V, kp, vp, table = _case(rng, T, Hq, Hkv, d, ps, roles)
        qb = int(rng.integers(0, T)) if trial % 3 == 0 else 0
        q = rng.standard_normal((T - qb, Hq, d))
        sink, window = int(rng.integers(0, 3)), int(rng.integers(0, 5))
        Ov, Lv = O.seg_paged_request(q, kp, vp, table, T, qb, roles, sink, window, 0.7, ps)
        Ob, Lb = O.brute_force_paged(q.tolist(), kp.tolist(), vp.tolist(), table.tolist(), T, qb,
                                     roles.tolist(), sink, window, 0.7, ps)
        assert np.allclose(Ov, np.array(Ob), atol=1e-12)
        assert np.allclose(Lv, np.array(Lb), atol=1e-12)


def _sdpa(q, K, V, G, mask, scale):
    qt = torch.from_numpy(q).permute(1, 0, 2)                        # [Hq, T, d]
    kt = torch.from_numpy(K).repeat_interleave(G, dim=0)             # [Hq, T, d]
    vt = torch.from_numpy(V).repeat_interleave(G, dim=0)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                            scale=scale).permute(1, 0, 2).numpy()


def test_global_heads_equal_causal_gqa_sdpa():
    """All-Global: causal attention of each query head against its KV
    group's keys (torch SDPA, fp64, K/V repeated per group)."""
    rng = np.random.default_rng(32)
    T, Hq, Hkv, d, ps = 37, 8, 2, 8, 8
    roles = np.ones(Hkv, np.uint8)
    K, V, kp, vp, table = _case(rng, T, Hq, Hkv, d, ps, roles)
    q = rng.standard_normal((T, Hq, d))
    scale = 1 / math.sqrt(d)
    Ov, Lv = O.seg_paged_request(q, kp, vp, table, T, 0, roles, 3, 4, scale, ps)
    mask = torch.tril(torch.ones(T, T, dtype=torch.bool))
    assert np.allclose(Ov, _sdpa(q, K, V, Hq // Hkv, mask, scale), atol=1e-12)
    sc = scale * torch.einsum("thd,hsd->hts", torch.from_numpy(q),
                              torch.from_numpy(K).repeat_interleave(Hq // Hkv, 0))
    sc = sc.masked_fill(~mask, float("-inf"))
    assert np.allclose(Lv, torch.logsumexp(sc, -1).T.numpy(), atol=1e-12)


def test_local_heads_equal_dense_plus_mask():
    """Local heads = dense attention over the whole prompt with a boolean
    mask that hides everything outside sink u [p - w, p] (the blog's "dense +
    mask" arm computes the same result)."""
    rng = np.random.default_rng(33)
    T, Hq, Hkv, d, ps = 45, 4, 2, 8, 4
    roles = np.zeros(Hkv, np.uint8)
    sink, window = 3, 6
    K, V, kp, vp, table = _case(rng, T, Hq, Hkv, d, ps, roles)
    q = rng.standard_normal((T, Hq, d))
    Ov, _ = O.seg_paged_request(q, kp, vp, table, T, 0, roles, sink, window, 0.4, ps)
    mask = torch.zeros(T, T, dtype=torch.bool)
    for p in range(T):
        for k in range(p + 1):
            mask[p, k] = k < sink or k >= p - window
    assert np.allclose(Ov, _sdpa(q, K, V, Hq // Hkv, mask, 0.4), atol=1e-12)


def test_physical_page_order_is_irrelevant():
    rng = np.random.default_rng(34)
    T, Hq, Hkv, d, ps = 30, 4, 2, 4, 4
    roles = np.array([0, 1], np.uint8)
    K, V, kp, vp, table = _case(rng, T, Hq, Hkv, d, ps, roles)
    q = rng.standard_normal((T, Hq, d))
    a = O.seg_paged_request(q, kp, vp, table, T, 0, roles, 2, 3, 0.5, ps)
    perm = rng.permutation(kp.shape[0])
    inv = np.argsort(perm)
    t2 = np.where(table >= 0, inv[np.maximum(table, 0)], -1)
    b = O.seg_paged_request(q, kp[perm], vp[perm], t2, T, 0, roles, 2, 3, 0.5, ps)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_local_heads_drop_pages_outside_sink_and_window():
    """The memory claim: a Local head that keeps only the pages its rows can
    see (sink and window) gives the same output; dropping a page it does need
    is caught."""
    rng = np.random.default_rng(35)
    T, Hq, Hkv, d, ps = 64, 4, 2, 4, 8
    roles = np.array([0, 1], np.uint8)
    sink, window = 2, 6
    K, V, kp, vp, table = _case(rng, T, Hq, Hkv, d, ps, roles)
    q = rng.standard_normal((1, Hq, d))
    p = T - 1   # decode row: the Local head needs block 0 (sink) and the last blocks
    full = O.seg_paged_request(q, kp, vp, table, T, p, roles, sink, window, 0.5, ps)
    t2 = table.copy()
    keep = {0} | set(range((p - window) // ps, p // ps + 1))
    for b in range(t2.shape[1]):
        if b not in keep:
            t2[0, b] = -1
    part = O.seg_paged_request(q, kp, vp, t2, T, p, roles, sink, window, 0.5, ps)
    assert np.array_equal(full[0], part[0]) and np.array_equal(full[1], part[1])
    t3 = t2.copy()
    t3[0, p // ps] = -1
    with pytest.raises(AssertionError):
        O.seg_paged_request(q, kp, vp, t3, T, p, roles, sink, window, 0.5, ps)


def _rope_complex(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """R(pos) on the last axis written with complex numbers: pair j (dims 2j,
    2j + 1) is the complex number x_2j + i x_2j+1 turned by exp(i pos theta_j),
    theta_j = base^(-2j/d).  An independent statement of the RoPE rotation."""
    d = x.shape[-1]
    theta = base ** (-2.0 * np.arange(d // 2) / d)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * pos[..., None] * theta)
    out = np.empty_like(x)
    out[..., 0::2] = z.real
    out[..., 1::2] = z.imag
    return out


@pytest.mark.parametrize("roles", [(1, 0), (0, 1)])
def test_relocated_documents_equal_keys_at_absolute_positions(roles):
    """Blog "Insight 1": a document cached alone (keys with RoPE at 0..n-1)
    and placed at offset delta attends exactly as if its keys had been
    computed at positions delta..delta+n-1.  Keys are built from raw vectors
    x_k both ways with the complex-number rotation; the oracle given the
    canonical pages and the block offsets must match the oracle given the
    absolute pages, and the opposite turn must not."""
    rng = np.random.default_rng(77)
    T, Hq, Hkv, d, ps, base = 40, 4, 2, 8, 8, 100.0
    delta = np.array([0, 0, 16, 16, 0])         # documents: blocks 0-1 at 0, 2-3 at 16; tail 4
    tok_delta = np.repeat(delta, ps)[:T]
    X = rng.standard_normal((Hkv, T, d))
    V = rng.standard_normal((Hkv, T, d))
    k_abs = _rope_complex(X, np.arange(T, dtype=np.float64)[None, :].repeat(Hkv, 0), base)
    k_can = _rope_complex(X, (np.arange(T) - tok_delta).astype(np.float64)[None, :].repeat(Hkv, 0),
                          base)
    nb = T // ps
    table = np.array([[g * nb + b for b in range(nb)] for g in range(Hkv)])

    def pages(K):
        return np.stack([K[g, b * ps:(b + 1) * ps] for g in range(Hkv) for b in range(nb)])

    q = rng.standard_normal((T, Hq, d)) * 2.0
    role = np.array(roles, np.uint8)
    args = (table, T, 0, role, 2, 6, 0.5, ps)
    O_ref, L_ref = O.seg_paged_request(q, pages(k_abs), pages(V), *args)
    O_rel, L_rel = O.seg_paged_request(q, pages(k_can), pages(V), *args, block_delta=delta,
                                       rope_base=base)
    assert np.abs(O_rel - O_ref).max() < 1e-12 and np.abs(L_rel - L_ref).max() < 1e-12
    O_bad, _ = O.seg_paged_request(q, pages(k_can), pages(V), *args, block_delta=-delta,
                                   rope_base=base)
    assert np.abs(O_bad - O_ref).max() > 1e-3


def test_zero_offsets_change_nothing():
    rng = np.random.default_rng(78)
    K, V, kp, vp, table = _case(rng, 23, 4, 2, 4, 4, None)
    q = rng.standard_normal((23, 4, 4))
    role = np.array([1, 0], np.uint8)
    a = O.seg_paged_request(q, kp, vp, table, 23, 0, role, 2, 5, 0.7, 4)
    b = O.seg_paged_request(q, kp, vp, table, 23, 0, role, 2, 5, 0.7, 4,
                            block_delta=np.zeros(table.shape[1], np.int64))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
