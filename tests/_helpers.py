"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI, evaluate the oracle on the same inputs, compare with the stated
tolerances."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
from position_independent_kv_gb300 import binding as B
from position_independent_kv_gb300.protected import build_bitmap
from position_independent_kv_gb300.workloads import make_workload

# Tolerances for bf16 inputs with fp32 accumulation against the fp64 oracle.
MAX_REL = 1e-2     # max |err| <= MAX_REL * max |ref|   (per tensor)
MEAN_REL = 2e-3    # sum |err| / sum |ref| <= MEAN_REL  (per tensor)
LSE_ABS = 1e-3     # |lse - lse_ref| <= LSE_ABS

# (label, stats) of every comparison made in this session; the conftest
# prints them at the end of the run so the margins to the bounds are visible.
PARITY_STATS: list = []


def record_stats(label: str, stats: dict, max_rel=MAX_REL, mean_rel=MEAN_REL, lse_abs=LSE_ABS):
    """Keep one comparison's error statistics with the bounds it was held to."""
    PARITY_STATS.append((label, dict(stats, max_bound=max_rel * stats["max_ref"],
                                     mean_bound=mean_rel, lse_bound=lse_abs)))


def run_gpu(wl, flags=0, stream=None):
    bm, prot_rows = build_bitmap(wl)
    plan = B.SegAttnPlan.from_workload(wl, bitmap=bm, flags=flags, stream=stream)
    ws = None
    if plan.workspace_bytes:
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=wl.q.device)
    out = wl.out_init.clone()
    lse = wl.lse_init.clone()
    plan.forward(wl.q, out, lse, ws, stream=stream)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    return out, lse, plan, bm, prot_rows


def sample_rows(req, prot: np.ndarray, rng: np.random.Generator, window: int, sink: int,
                cap: int = 96) -> np.ndarray:
    """Stratified rows: segment edges, window edges that cross a segment
    boundary, sink edges, random protected and unprotected rows, the last."""
    T, qb = req.T, req.q_row_begin
    pick = {T - 1, qb}
    for s in req.segments:
        for p in (s.delta, s.delta + 1, s.delta + s.n - 1, s.delta + min(window, s.n - 1),
                  s.delta + window + 1):
            pick.add(p)
    pick |= {sink - 1, sink, sink + 1, window, window + 1, window + sink + 1}
    pick = {p for p in pick if qb <= p < T}
    allr = np.arange(qb, T)
    pr = allr[prot[qb:]]
    up = allr[~prot[qb:]]
    if len(pr):
        pick |= set(rng.choice(pr, size=min(16, len(pr)), replace=False).tolist())
    if len(up):
        pick |= set(rng.choice(up, size=min(16, len(up)), replace=False).tolist())
    rows = np.array(sorted(pick), dtype=np.int64)
    if len(rows) > cap:
        keep = rng.choice(len(rows), size=cap, replace=False)
        rows = np.sort(rows[keep])
    return rows


def oracle_rows(wl, prot_rows, rows_per_req=None):
    """Oracle O/lse for the requested rows of every request (all rows when
    rows_per_req is None).  Returns lists of (flat_row_indices, O, lse)."""
    res = []
    offs = wl.row_offsets()
    for r, req in enumerate(wl.requests):
        segs = [(s.latent.double().cpu().numpy(), s.delta, s.is_new) for s in req.segments]
        rows = (np.arange(req.q_row_begin, req.T) if rows_per_req is None
                else np.asarray(rows_per_req[r], dtype=np.int64))
        flat = offs[r] + (rows - req.q_row_begin)
        fl = torch.from_numpy(flat).to(wl.q.device)
        q = wl.q[fl].double().cpu().numpy()
        oi = wl.out_init[fl].double().cpu().numpy()
        li = wl.lse_init[fl].double().cpu().numpy()
        Oo, Lo = O.seg_attn_request(q, segs, req.T, req.q_row_begin, wl.head_role, wl.d_nope,
                                    wl.rope_base, wl.scale, wl.sink, wl.window, prot_rows[r],
                                    oi, li, rows=rows, sampled=True, v_rope=wl.v_rope)
        res.append((flat, Oo, Lo))
    return res


def computed_mask(wl, prot_rows, flat_rows_per_req, rows_per_req):
    """bool [n, H]: which (row, head) the method recomputes."""
    out = []
    glob = wl.head_role.astype(bool)
    for r, req in enumerate(wl.requests):
        rows = np.asarray(rows_per_req[r])
        m = np.zeros((len(rows), wl.H), dtype=bool)
        m[:, glob] = True
        m[:, ~glob] = prot_rows[r][rows][:, None] | _new_rows(req)[rows][:, None]
        out.append(m)
    return out


def _new_rows(req):
    new = np.zeros(req.T, dtype=bool)
    for s in req.segments:
        if s.is_new:
            new[s.delta:s.delta + s.n] = True
    return new


def compare(wl, out, lse, prot_rows, ref, rows_per_req, label=""):
    """Tolerance check on recomputed (row, head) pairs and bit-exact check on
    the untouched ones, for the rows the oracle evaluated."""
    go_all, ro_all, gl_all, rl_all = [], [], [], []
    for r, (flat, Oo, Lo) in enumerate(ref):
        fl = torch.from_numpy(flat).to(out.device)
        go = out[fl].double().cpu().numpy()
        gl = lse[fl].double().cpu().numpy()
        cm = computed_mask(wl, prot_rows, None, rows_per_req)[r]
        oi = wl.out_init[fl].cpu()
        li = wl.lse_init[fl].cpu()
        # untouched pairs keep their bytes
        un = torch.from_numpy(~cm)
        assert torch.equal(out[fl].cpu()[un], oi[un]), f"{label}: untouched output changed"
        assert torch.equal(lse[fl].cpu()[un], li[un]), f"{label}: untouched lse changed"
        go_all.append(go[cm])
        ro_all.append(Oo[cm])
        gl_all.append(gl[cm])
        rl_all.append(Lo[cm])
    go = np.concatenate(go_all)
    ro = np.concatenate(ro_all)
    gl = np.concatenate(gl_all)
    rl = np.concatenate(rl_all)
    err = np.abs(go - ro)
    stats = dict(max_err=float(err.max()), max_ref=float(np.abs(ro).max()),
                 mean_rel=float(err.sum() / np.abs(ro).sum()),
                 lse_err=float(np.abs(gl - rl).max()), n=int(go.shape[0]))
    record_stats(label, stats)
    assert np.isfinite(go).all() and np.isfinite(gl).all(), f"{label}: non-finite output"
    assert stats["max_err"] <= MAX_REL * stats["max_ref"], f"{label}: {stats}"
    assert stats["mean_rel"] <= MEAN_REL, f"{label}: {stats}"
    assert stats["lse_err"] <= LSE_ABS, f"{label}: {stats}"
    return stats


def untouched_all_rows(wl, out, lse, prot_rows):
    """Bit-exact check over EVERY row: unrecomputed Local pairs keep their
    cached bytes and their lse sentinel; recomputed pairs got a real lse."""
    offs = wl.row_offsets()
    loc = torch.from_numpy(~wl.head_role.astype(bool)).to(out.device)
    for r, req in enumerate(wl.requests):
        n = req.n_computed
        pr = torch.from_numpy((prot_rows[r] | _new_rows(req))[req.q_row_begin:]).to(out.device)
        sl = slice(offs[r], offs[r] + n)
        un = (~pr)[:, None] & loc[None, :]
        o, oi = out[sl], wl.out_init[sl]
        l, li = lse[sl], wl.lse_init[sl]
        assert torch.equal(o[un], oi[un])
        assert torch.equal(l[un], li[un])
        assert bool((l[~un] != li[~un]).all()), "a recomputed pair kept the lse sentinel"
