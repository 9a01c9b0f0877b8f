"""CPU fp64 oracle for SegPagedAttention on grouped-query attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA
path and imports nothing from the product package.

What it computes (RedKnot blog, "Insight 3: savings must show up in memory"
and "Insight 1"): the KV cache is stored per KV head in pages; a Global head
keeps the pages of the whole prompt, a Local head only those of its sink and
window.  Attention itself is unchanged: every query head of a KV group sees
the keys of that KV head that its role makes visible -- Global: every k <= p;
Local: k <= p with k < sink or k >= p - w (blog, the window W(i) and its
worked example) -- and the page layout only decides which keys are touched.

Readings: a page holds `page_size` consecutive tokens of ONE KV head (logical
block b of a sequence covers tokens [b * page_size, (b + 1) * page_size));
`block_table[r][g][b]` is the physical page of block b of KV head g in request
r, or -1 where the head keeps no page; query head i belongs to KV head
i // (Hq / Hkv); keys already carry their RoPE at absolute positions; every
computed row p of every query head is evaluated.  The visibility rule and the
dense softmax are the ones of `seg_attn` (imported, so both oracles read the
blog's window rule one way).

Relocated documents (`block_delta`): a document cached alone has its keys'
RoPE at positions 0..n-1; placed at request offset delta, its pages are
reused as they are.  Reading: `block_delta[b]` is the offset of the document
that logical block b belongs to (every KV head alike), so a key stored at
absolute token k of block b carries its RoPE at position k - block_delta[b].
The oracle relocates each such key physically, K(k) = R(delta) K_stored
(blog "Insight 1", the relocation equation K(p_new) = R(p_new) R(p_old)^-1
K(p_old)), with RoPE on all head dims as interleaved pairs, theta_j =
base^(-2j/d) (the `rotate` of `seg_attn`), and then attends as above.
"""
from __future__ import annotations

import numpy as np

from .seg_attn import attend, rotate, visible_keys


def gather_head(pages: np.ndarray, table_row, n_tokens: int, page_size: int, need=None):
    """Logical [n_tokens, d] keys (or values) of one KV head from its pages.
    Blocks without a page (-1) are NaN; `need` (bool [n_tokens]) asserts that
    every needed token has a page."""
    d = pages.shape[-1]
    out = np.full((n_tokens, d), np.nan)
    for b in range((n_tokens + page_size - 1) // page_size):
        pg = int(table_row[b]) if b < len(table_row) else -1
        lo, hi = b * page_size, min(n_tokens, (b + 1) * page_size)
        if pg >= 0:
            out[lo:hi] = pages[pg, :hi - lo]
        elif need is not None:
            assert not need[lo:hi].any(), f"block {b} is needed but has no page"
    return out


def relocate_blocks(K: np.ndarray, block_delta, page_size: int, base: float) -> np.ndarray:
    """K [T, d] of one KV head with every key of block b moved from its stored
    RoPE position k - block_delta[b] to its absolute position k: R(+delta)."""
    T = K.shape[0]
    pos = np.array([block_delta[k // page_size] for k in range(T)], dtype=np.float64)
    return rotate(K, pos, base)


def seg_paged_request(q: np.ndarray, k_pages: np.ndarray, v_pages: np.ndarray,
                      table: np.ndarray, T: int, q_row_begin: int, kv_role, sink: int,
                      window: int, scale: float, page_size: int, rows=None, sampled=False,
                      block_delta=None, rope_base: float = 10000.0):
    """One request.

    q         fp64 [T - q_row_begin, Hq, d]  (row i = absolute row q_row_begin + i)
    k_pages   fp64 [pages, page_size, d]; v_pages likewise
    table     int [Hkv, max_blocks]  physical page of each logical block, -1 = none
    kv_role   [Hkv] 0 Local, 1 Global
    rows      absolute rows to evaluate (default every computed row); with
              `sampled` q holds only those rows, in that order.
    block_delta  optional [max_blocks] document offset of each logical block
              (keys stored with RoPE at k - delta); rope_base its RoPE base.

    Returns O [n_rows, Hq, d], lse [n_rows, Hq]."""
    kv_role = np.asarray(kv_role).astype(bool)
    Hkv = len(kv_role)
    Hq = q.shape[1]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    if rows is None:
        rows = np.arange(q_row_begin, T)
    rows = np.asarray(rows, dtype=np.int64)
    # tokens each KV head must have: the union of the visible sets of the rows
    need = np.zeros((Hkv, T), dtype=bool)
    for p in rows:
        for g in range(Hkv):
            need[g, visible_keys(int(p), bool(kv_role[g]), sink, window)] = True
    K = [gather_head(k_pages, table[g], T, page_size, need[g]) for g in range(Hkv)]
    if block_delta is not None:
        K = [relocate_blocks(k, block_delta, page_size, rope_base) for k in K]
    V = [gather_head(v_pages, table[g], T, page_size) for g in range(Hkv)]
    d = q.shape[2]
    O = np.empty((len(rows), Hq, d))
    L = np.empty((len(rows), Hq))
    for i, p in enumerate(rows):
        assert q_row_begin <= p < T
        r = i if sampled else p - q_row_begin
        for g in range(Hkv):
            keys = visible_keys(int(p), bool(kv_role[g]), sink, window)
            heads = slice(g * G, (g + 1) * G)
            o, l = attend(q[r, heads], K[g][keys], V[g][keys], scale)
            O[i, heads], L[i, heads] = o, l
    return O, L


def brute_force_paged(q, k_pages, v_pages, table, T, q_row_begin, kv_role, sink, window,
                      scale, page_size):
    """Pure-Python loops (no NumPy arithmetic) over the pages themselves, for
    tiny shapes: the same contract as seg_paged_request on nested lists."""
    import math
    Hkv = len(kv_role)
    Hq = len(q[0])
    G = Hq // Hkv
    d = len(q[0][0])
    O, L = [], []
    for p in range(q_row_begin, T):
        r = p - q_row_begin
        orow, lrow = [], []
        for i in range(Hq):
            g = i // G
            keys = [k for k in range(p + 1)
                    if kv_role[g] or k < sink or k >= p - window]
            xs, vs = [], []
            for k in keys:
                pg = table[g][k // page_size]
                kv = k_pages[pg][k % page_size]
                xs.append(scale * sum(q[r][i][c] * kv[c] for c in range(d)))
                vs.append(v_pages[pg][k % page_size])
            mx = max(xs)
            es = [math.exp(x - mx) for x in xs]
            den = sum(es)
            orow.append([sum(es[j] * vs[j][c] for j in range(len(keys))) / den for c in range(d)])
            lrow.append(mx + math.log(den))
        O.append(orow)
        L.append(lrow)
    return O, L
