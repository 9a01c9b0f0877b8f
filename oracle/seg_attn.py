"""CPU fp64 oracle for segment-relocated MLA attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA
path and imports nothing from the product package.

What it computes is the plain definition of the method, written out in the
order the pages give it:

1. Relocation.  A document built alone at positions 0..n-1 and placed at
   request offset delta has its keys moved to absolute positions by the RoPE
   rotation K(p_new) = R(p_new) R(p_old)^-1 K(p_old) (RedKnot blog,
   "Insight 1", the relocation equation), i.e. every canonical k_rope row j is
   rotated by R(delta) to sit at position delta + j.  The RedKnot-MLA paper
   (RoPE-orthogonality paragraph) states that rotating the query by -delta
   instead gives the same scores; the oracle does the physical rotation.
2. Concatenation into one [T, d_nope + d_rope] key matrix; V = the c_nope
   columns of the same rows (MLA's shared packed latent, paper first
   paragraphs).
3. Visibility.  Global heads: every key k <= p (recomputed in full, blog
   "Insight 1" rule 1).  Local heads: sink union [p - w, p]
   (blog "Insight 1", the window W(i) and its worked example).
4. Dense softmax attention per head in fp64: x = s q.K, O = softmax(x) V,
   lse = max x + ln sum exp(x - max x).
5. Assembly.  Global heads keep every computed row; Local heads are replaced
   only on protected rows; all other Local rows keep the cached values
   unchanged (paper, protected-set paragraph: "replaced, never double
   counted").

Readings where the pages are silent are listed with the functions below.
Every function here is pinned by `tests/test_oracle_pins.py` against closed
forms, library routines or brute force.
"""
from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------
# RoPE (RedKnot-MLA paper, RoPE-orthogonality paragraph; RedKnot blog,
# "Insight 1" relocation equation).  Reading: interleaved pairs (2k, 2k+1) of
# the rope slice, theta_k = base^(-2k/d_rope), angle = position * theta_k,
# R(phi) maps (x, y) -> (x cos phi - y sin phi, x sin phi + y cos phi).
# --------------------------------------------------------------------------


def rope_theta(d_rope: int, base: float) -> np.ndarray:
    k = np.arange(d_rope // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * k / d_rope)


def rotate(x: np.ndarray, pos, base: float) -> np.ndarray:
    """R(pos) applied to the last axis of x (fp64).  pos broadcasts against
    x[..., 0]; negative positions rotate backwards."""
    x = np.asarray(x, dtype=np.float64)
    d_rope = x.shape[-1]
    theta = rope_theta(d_rope, base)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta
    c, s = np.cos(ang), np.sin(ang)
    xe, xo = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = xe * c - xo * s
    out[..., 1::2] = xe * s + xo * c
    return out


# --------------------------------------------------------------------------
# Relocation + concatenation (steps 1-2)
# --------------------------------------------------------------------------


def relocate(segments, T: int, d_nope: int, base: float):
    """segments: iterable of (latent fp64 [n, d_k], delta).  Returns K_full
    [T, d_k] with every row at its absolute position and V_full [T, d_nope].

    Reading: the new rows of the request are one more segment, canonical at
    0..n_new-1 and placed at its own offset, so they relocate the same way."""
    segments = list(segments)
    d_k = segments[0][0].shape[1]
    K = np.zeros((T, d_k), dtype=np.float64)
    filled = np.zeros(T, dtype=bool)
    for lat, delta in segments:
        lat = np.asarray(lat, dtype=np.float64)
        n = lat.shape[0]
        if n == 0:
            continue
        assert 0 <= delta and delta + n <= T, "segment outside the request"
        assert not filled[delta:delta + n].any(), "segments overlap"
        K[delta:delta + n, :d_nope] = lat[:, :d_nope]
        K[delta:delta + n, d_nope:] = rotate(lat[:, d_nope:], float(delta), base)
        filled[delta:delta + n] = True
    assert filled.all(), "segments do not cover the request"
    return K, K[:, :d_nope]


# --------------------------------------------------------------------------
# Visibility (step 3).  Readings: causal diagonal included (k <= p); the sink
# is request-absolute positions 0..sink-1; the window is [p - w, p] inclusive
# (w + 1 keys) clipped at 0; the union has no duplicates.
# --------------------------------------------------------------------------


def visible_keys(p: int, is_global: bool, sink: int, window: int) -> np.ndarray:
    if is_global:
        return np.arange(p + 1)
    lo = max(0, p - window)
    if lo <= sink:
        return np.arange(p + 1)
    return np.concatenate([np.arange(min(sink, p + 1)), np.arange(lo, p + 1)])


# --------------------------------------------------------------------------
# Dense softmax attention (step 4).  Reading: natural-log LSE of the scaled
# scores.
# --------------------------------------------------------------------------


def attend(qh: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """qh [h, d_k] against all rows of K/V.  Returns O [h, d_v], lse [h]."""
    x = scale * (qh @ K.T)
    m = x.max(axis=1, keepdims=True)
    e = np.exp(x - m)
    l = e.sum(axis=1, keepdims=True)
    o = (e @ V) / l
    return o, m[:, 0] + np.log(l[:, 0])


def seg_attn_request(q: np.ndarray, segments, T: int, q_row_begin: int,
                     head_role, d_nope: int, base: float, scale: float,
                     sink: int, window: int, protected: np.ndarray,
                     out_init: np.ndarray, lse_init: np.ndarray, rows=None, sampled=False,
                     v_rope: bool = False):
    """One request.

    q         fp64 [T - q_row_begin, H, d_k]  (row i = absolute row q_row_begin + i)
    segments  list of (latent fp64 [n, d_k], delta, is_new)
    protected bool [T]  protected rows (new rows are added here as well)
    out_init  [T - q_row_begin, H, d_nope] cached values;  lse_init likewise
    rows      absolute rows to evaluate (default: every computed row)
    sampled   if True, q / out_init / lse_init hold only the evaluated rows,
              in the order of `rows`
    v_rope    the value carries a rotary part (output-phase restore, see
              `restore_output_phase`): V is the whole relocated key row, so
              out_init and the result have d_k columns

    Returns (O, lse) for the evaluated rows, already assembled: Global heads
    computed, Local heads computed on protected rows and copied otherwise.
    """
    K, V = relocate([(lat, d) for lat, d, _ in segments], T, d_nope, base)
    if v_rope:
        V = K
    prot = np.array(protected, dtype=bool).copy()
    for lat, d, is_new in segments:
        if is_new:
            prot[d:d + np.asarray(lat).shape[0]] = True
    role = np.asarray(head_role).astype(bool)
    gh = np.nonzero(role)[0]
    lh = np.nonzero(~role)[0]
    if rows is None:
        rows = np.arange(q_row_begin, T)
    rows = np.asarray(rows, dtype=np.int64)
    H = q.shape[1]
    O = np.empty((len(rows), H, V.shape[1]), dtype=np.float64)
    L = np.empty((len(rows), H), dtype=np.float64)
    for i, p in enumerate(rows):
        assert q_row_begin <= p < T
        r = i if sampled else p - q_row_begin
        O[i] = out_init[r]
        L[i] = lse_init[r]
        if len(gh):
            o, l = attend(q[r, gh], K[:p + 1], V[:p + 1], scale)
            if v_rope:
                o = restore_output_phase(o, int(p), d_nope, base)
            O[i, gh], L[i, gh] = o, l
        if len(lh) and prot[p]:
            keys = visible_keys(int(p), False, sink, window)
            o, l = attend(q[r, lh], K[keys], V[keys], scale)
            if v_rope:
                o = restore_output_phase(o, int(p), d_nope, base)
            O[i, lh], L[i, lh] = o, l
    return O, L


# --------------------------------------------------------------------------
# Output-phase restore (RedKnot-MLA paper: the head-partition paragraph
# defines the inverse output RoPE R^-1 applied to the attention output before
# the sliced W_a; the RoPE-orthogonality paragraph: after attending the
# canonical latent the runtime "restores the output phase").  Reading: when
# the value is the packed latent row itself, its rope slice carries the key's
# absolute phase R(k) once relocated (step 1), so the output's rope slice is
# sum_k P_k R(k) v_k; the inverse output RoPE at the query's absolute
# position p turns it by R(-p), leaving sum_k P_k R(k - p) v_k, which depends
# on relative positions only.
# --------------------------------------------------------------------------


def restore_output_phase(o: np.ndarray, p: int, d_nope: int, base: float) -> np.ndarray:
    """o [..., d_k] computed against relocated values -> the same with the
    rope slice turned by R(-p)."""
    o = np.array(o, dtype=np.float64, copy=True)
    o[..., d_nope:] = rotate(o[..., d_nope:], -float(p), base)
    return o


# --------------------------------------------------------------------------
# Segment LSE merge (paper, RoPE-orthogonality paragraph: "combines segment
# statistics with a numerically stable log-sum-exp merge").  Reading: parts
# with lse = -inf carry weight 0; if every part is -inf the result is O = 0,
# lse = -inf.
# --------------------------------------------------------------------------


def lse_merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """o_parts [P, ..., d_v], lse_parts [P, ...] -> (O [..., d_v], lse [...])."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - m_safe[None]), 0.0)
    s = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, s, 1.0)), -np.inf)
    o = np.where(finite[..., None],
                 (w[..., None] * o_parts).sum(axis=0) / np.where(finite, s, 1.0)[..., None],
                 0.0)
    return o, lse


def attend_partial(qh: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Per-part statistics for the merge: an empty part gives O = 0, lse = -inf."""
    if K.shape[0] == 0:
        return np.zeros((qh.shape[0], V.shape[1])), np.full(qh.shape[0], -np.inf)
    return attend(qh, K, V, scale)


# --------------------------------------------------------------------------
# Protected-row set (paper, protected-set paragraph: A = Q u N u D u B128 u
# I_top u T32K, budget 10/20/25 %).  Readings: B_b = rows [0, min(b, n)) and
# [max(0, n - b), n) of every cached segment; Indexer rows are stood in for
# by the seeded draws `u` (Bernoulli rule) and `perm` (budget rule); the
# budget target is ceil(pct * C / 100) over the C cached rows, boundary rows
# first, then non-boundary cached rows in `perm` order; new rows are always
# protected on top.
# --------------------------------------------------------------------------


def build_protected(T: int, segs, boundary: int, p_random: float, budget: float,
                    none: bool, u: np.ndarray, perm: np.ndarray, dirty=None) -> np.ndarray:
    """segs: list of (n, delta, is_new).  dirty: optional bool [T] of rows
    whose cached values are stale (the paper's D); they are protected on top
    of the rule and do not count toward the budget.  Returns bool [T]."""
    prot = [False] * T
    cached = [False] * T
    bnd = [False] * T
    for n, d, is_new in segs:
        for j in range(n):
            if is_new:
                prot[d + j] = True
            else:
                cached[d + j] = True
                if j < boundary or j >= n - boundary:
                    bnd[d + j] = True
    if not none:
        if p_random > 0:
            for p in range(T):
                if cached[p] and (bnd[p] or u[p] < p_random):
                    prot[p] = True
        elif budget > 0:
            C = sum(cached)
            pct = int(round(budget * 100))
            target = -(-pct * C // 100)
            chosen = sum(bnd)
            for p in range(T):
                if bnd[p]:
                    prot[p] = True
            for p in perm:
                if chosen >= target:
                    break
                p = int(p)
                if cached[p] and not bnd[p]:
                    prot[p] = True
                    chosen += 1
        else:
            for p in range(T):
                if bnd[p]:
                    prot[p] = True
    if dirty is not None:
        for p in range(T):
            if dirty[p]:
                prot[p] = True
    return np.array(prot, dtype=bool)


def bitmap_words(prot: np.ndarray) -> np.ndarray:
    """bool [T] -> uint32 words, bit p%32 of word p//32 (LSB first)."""
    T = len(prot)
    words = np.zeros((T + 31) // 32, dtype=np.uint32)
    for p in range(T):
        if prot[p]:
            words[p // 32] |= np.uint32(1) << np.uint32(p % 32)
    return words


# --------------------------------------------------------------------------
# Pure-Python brute force for tiny shapes (no NumPy in the arithmetic).
# --------------------------------------------------------------------------


def brute_force(q, segments, T, q_row_begin, head_role, d_nope, base, scale,
                sink, window, protected, out_init, lse_init, v_rope=False):
    """Same contract as seg_attn_request on nested Python lists, every row."""
    d_k = len(q[0][0])
    d_rope = d_k - d_nope
    Kf = [None] * T
    for lat, delta, _ in segments:
        for j, row in enumerate(lat):
            p = delta + j
            k = list(row[:d_nope])
            for i in range(d_rope // 2):
                th = float(base) ** (-2.0 * i / d_rope)
                a = delta * th
                x, y = row[d_nope + 2 * i], row[d_nope + 2 * i + 1]
                k += [x * math.cos(a) - y * math.sin(a), x * math.sin(a) + y * math.cos(a)]
            Kf[p] = k
    prot = list(protected)
    for lat, delta, is_new in segments:
        if is_new:
            for j in range(len(lat)):
                prot[delta + j] = True
    H = len(q[0])
    O, L = [], []
    for p in range(q_row_begin, T):
        r = p - q_row_begin
        orow, lrow = [], []
        for h in range(H):
            g = bool(head_role[h])
            if not g and not prot[p]:
                orow.append(list(out_init[r][h]))
                lrow.append(lse_init[r][h])
                continue
            keys = []
            for k in range(p + 1):
                if g or k < sink or k >= p - window:
                    keys.append(k)
            xs = [scale * sum(q[r][h][c] * Kf[k][c] for c in range(d_k)) for k in keys]
            mx = max(xs)
            es = [math.exp(x - mx) for x in xs]
            den = sum(es)
            d_v = d_k if v_rope else d_nope
            ov = [sum(es[i] * Kf[k][c] for i, k in enumerate(keys)) / den for c in range(d_v)]
            if v_rope:  # inverse output RoPE at the query's own position
                for i in range(d_rope // 2):
                    a = -p * float(base) ** (-2.0 * i / d_rope)
                    x, y = ov[d_nope + 2 * i], ov[d_nope + 2 * i + 1]
                    ov[d_nope + 2 * i] = x * math.cos(a) - y * math.sin(a)
                    ov[d_nope + 2 * i + 1] = x * math.sin(a) + y * math.cos(a)
            orow.append(ov)
            lrow.append(mx + math.log(den))
        O.append(orow)
        L.append(lrow)
    return O, L
