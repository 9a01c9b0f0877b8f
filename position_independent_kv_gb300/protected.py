"""Protected-row set of RedKnot-MLA (host side, vectorised).

RedKnot-MLA paper (arXiv 2609.07008), protected-set paragraph: the protected
token-row set is the union of the query rows Q, the new rows N, dirty rows
D, the first and last 128 rows of every relocated segment B_128, rows the
Indexer selects I_top and the recent 32K tail T_32K; a fixed controller may
widen it to 10 %, 20 % or 25 % of the candidate rows.  Cached Local values on
these rows are replaced by recomputed ones.

The Indexer needs trained weights, so its rows are stood in for by the seeded
draws that `workloads` supplies: an independent uniform per row (Bernoulli
rule, p_random) or a row permutation (budget rule).  Conventions:

* B_b = rows [0, min(b, n)) and [max(0, n - b), n) of every cached segment;
* budget target = ceil(pct * C / 100) over the C cached rows (integer
  arithmetic, pct = round(100 * budget)); boundary rows first, then
  non-boundary cached rows in permutation order until the target is reached;
  if the boundary rows alone exceed the target they are all kept;
* new rows (the request's query rows and, for the long-context workload, the
  recomputed 32K tail) are always protected.

The result is a bitmap of uint32 words per request, bit p % 32 of word
p // 32 set when absolute row p is protected (LSB first).
"""
from __future__ import annotations

import numpy as np

from .workloads import ProtectRule, Request


def protected_rows(req: Request, rule: ProtectRule) -> np.ndarray:
    T = req.T
    prot = np.zeros(T, dtype=bool)
    cached = np.zeros(T, dtype=bool)
    bnd = np.zeros(T, dtype=bool)
    for s in req.segments:
        if s.is_new:
            prot[s.delta:s.delta + s.n] = True
            continue
        cached[s.delta:s.delta + s.n] = True
        b = min(rule.boundary, s.n)
        bnd[s.delta:s.delta + b] = True
        bnd[s.delta + max(0, s.n - rule.boundary):s.delta + s.n] = True
    if rule.none:
        return prot
    if rule.p_random > 0:
        prot |= cached & (bnd | (req.u < rule.p_random))
    elif rule.budget > 0:
        C = int(cached.sum())
        pct = int(round(rule.budget * 100))
        target = -(-pct * C // 100)
        prot |= bnd
        need = target - int(bnd.sum())
        if need > 0:
            cand = req.perm[(cached & ~bnd)[req.perm]]
            prot[cand[:need]] = True
    else:
        prot |= bnd
    return prot


def pack_bits(prot: np.ndarray) -> np.ndarray:
    T = prot.shape[0]
    nw = (T + 31) // 32
    padded = np.zeros(nw * 32, dtype=np.uint64)
    padded[:T] = prot.astype(np.uint64)
    weights = (np.uint64(1) << np.arange(32, dtype=np.uint64))
    return (padded.reshape(nw, 32) * weights).sum(axis=1).astype(np.uint32)


def build_bitmap(wl) -> tuple[np.ndarray, list[np.ndarray]]:
    """Concatenated per-request bitmap words and the per-request bool rows."""
    words, rows = [], []
    for req in wl.requests:
        p = protected_rows(req, wl.rule)
        rows.append(p)
        words.append(pack_bits(p))
    return np.concatenate(words) if words else np.zeros(0, np.uint32), rows
