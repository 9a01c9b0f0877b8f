"""GPU parity: the CUDA path, called through the C ABI, against the fp64
oracle on the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from _helpers import (LSE_ABS, compare, oracle_rows, run_gpu, sample_rows,
                      untouched_all_rows)
from position_independent_kv_gb300 import binding as B
from position_independent_kv_gb300 import build as BUILD
from position_independent_kv_gb300.protected import build_bitmap
from position_independent_kv_gb300.workloads import SPECS, make_workload

pytestmark = pytest.mark.gpu

MINI = ["tiny", "tiny_wide", "flash_mini", "varlen_mini", "ctx128k_mini", "decode_mini"]
KERNELS = {"default": 0, "cta_pair": B.RK_PLAN_CTA_PAIR, "single_cta": B.RK_PLAN_SINGLE_CTA,
           "legacy": B.RK_PLAN_LEGACY_MMA}


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BUILD.build()


def _sharp(name):
    s = SPECS[name]
    return 4.0 * (s.d_nope + s.d_rope)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("sharp", [False, True], ids=["stated", "sharp"])
@pytest.mark.parametrize("name", MINI)
def test_parity_every_row(name, sharp, kernel):
    """Every computed row of the reduced workloads, both the stated input
    distribution and a sharp one (score std ~4) that makes the relocation
    decisive."""
    wl = make_workload(name, seed=0, device="cuda", q_scale=_sharp(name) if sharp else 1.0)
    out, lse, plan, bm, prot = run_gpu(wl, flags=KERNELS[kernel])
    ref = oracle_rows(wl, prot)
    rows = [np.arange(r.q_row_begin, r.T) for r in wl.requests]
    compare(wl, out, lse, prot, ref, rows, label=f"{name}/{kernel}/{sharp}")
    untouched_all_rows(wl, out, lse, prot)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("name", MINI + ["flash", "decode"])
def test_visible_key_counts_exact(name, kernel):
    """With q = 0 every visible key scores 0, so exp(lse) is exactly the
    number of visible keys: checks the masks bit-exactly on every computed
    (row, head) pair against the oracle's visibility rule."""
    wl = make_workload(name, seed=0, device="cuda")
    wl.q.zero_()
    out, lse, plan, bm, prot = run_gpu(wl, flags=KERNELS[kernel])
    offs = wl.row_offsets()
    glob = wl.head_role.astype(bool)
    for r, req in enumerate(wl.requests):
        p = np.arange(req.q_row_begin, req.T)
        l = lse[offs[r]:offs[r] + len(p)].double().cpu().numpy()
        cnt = np.rint(np.exp(np.minimum(l, 700.0)))
        assert np.array_equal(cnt[:, glob], np.broadcast_to((p + 1)[:, None], cnt[:, glob].shape))
        new = np.zeros(req.T, bool)
        for s in req.segments:
            if s.is_new:
                new[s.delta:s.delta + s.n] = True
        pr = (prot[r] | new)[req.q_row_begin:]
        if (~glob).any() and pr.any():
            want = np.array([len(O.visible_keys(int(x), False, wl.sink, wl.window))
                             for x in p[pr]], dtype=np.float64)
            assert np.array_equal(cnt[pr][:, ~glob],
                                  np.broadcast_to(want[:, None], cnt[pr][:, ~glob].shape))


def test_decisive_relocation_probe():
    """Queries aimed at one relocated key of another segment (q_rope =
    c * R(delta_i) k_rope_j): the probe key must dominate on the GPU exactly
    as in the oracle."""
    wl = make_workload("flash_mini", seed=1, device="cuda")
    req = wl.requests[0]
    rng = np.random.default_rng(0)
    glob = np.nonzero(wl.head_role)[0]
    targets = []
    for _ in range(24):
        p = int(rng.integers(300, req.T))
        cands = [s for s in req.segments if s.delta > 0 and s.delta < p and not s.is_new]
        if not cands:
            continue
        s = cands[int(rng.integers(0, len(cands)))]
        j = int(rng.integers(0, min(s.n, p - s.delta)))
        h = int(glob[int(rng.integers(0, len(glob)))])
        kr = s.latent[j, wl.d_nope:].double().cpu().numpy()
        qr = O.rotate(kr, float(s.delta), wl.rope_base)
        qr = qr * (12.0 / (wl.scale * float(kr @ kr)))
        wl.q[p, h] = 0
        wl.q[p, h, wl.d_nope:] = torch.from_numpy(qr).to(torch.bfloat16).cuda()
        targets.append((p, h))
    out, lse, plan, bm, prot = run_gpu(wl)
    rows = [np.array(sorted({p for p, _ in targets}))]
    ref = oracle_rows(wl, prot, rows)
    compare(wl, out, lse, prot, ref, rows, label="probe")
    flat, Oo, Lo = ref[0]
    for p, h in targets:
        i = int(np.nonzero(rows[0] == p)[0][0])
        assert Lo[i, h] > 10.0   # the probe dominates in the oracle too


@pytest.mark.parametrize("name", ["flash", "varlen", "ctx128k", "decode"])
def test_parity_full_size_sampled(name):
    """Full benchmark sizes in the benchmark's launch configuration: sampled
    rows against the oracle, every row for the untouched-bytes check."""
    wl = make_workload(name, seed=0, device="cuda")
    out, lse, plan, bm, prot = run_gpu(wl)
    rng = np.random.default_rng(11)
    cap = 6 if name == "decode" else 72
    rows = [sample_rows(req, prot[r], rng, wl.window, wl.sink, cap=cap)
            for r, req in enumerate(wl.requests)]
    ref = oracle_rows(wl, prot, rows)
    compare(wl, out, lse, prot, ref, rows, label=name)
    untouched_all_rows(wl, out, lse, prot)


def test_replacement_independent_of_cached_values():
    """Recomputed pairs do not depend on the pre-filled cache (replaced,
    never added); untouched pairs keep whichever cache was there."""
    wl = make_workload("flash_mini", seed=2, device="cuda")
    out1, lse1, plan, bm, prot = run_gpu(wl)
    wl.out_init = torch.randn_like(wl.out_init, dtype=torch.float32).to(torch.bfloat16)
    wl.lse_init = torch.full_like(wl.lse_init, -7.0)
    out2, lse2, *_ = run_gpu(wl)
    new = np.zeros(wl.requests[0].T, bool)
    for s in wl.requests[0].segments:
        if s.is_new:
            new[s.delta:s.delta + s.n] = True
    pr = torch.from_numpy(prot[0] | new).cuda()
    glob = torch.from_numpy(wl.head_role.astype(bool)).cuda()
    comp = pr[:, None] | glob[None, :]
    assert torch.equal(out1[comp], out2[comp]) and torch.equal(lse1[comp], lse2[comp])
    assert torch.equal(out2[~comp], wl.out_init[~comp])


def test_plan_reuse_and_stream():
    """One plan, two forwards with different queries, on a side stream."""
    wl = make_workload("varlen_mini", seed=3, device="cuda")
    bm, prot = build_bitmap(wl)
    s = torch.cuda.Stream()
    plan = B.SegAttnPlan.from_workload(wl, bitmap=bm, stream=s)
    for it in range(2):
        if it:
            wl.q = (torch.randn(wl.q.shape, device="cuda") * 2 / math.sqrt(wl.d_k)).to(torch.bfloat16)
        out, lse = wl.out_init.clone(), wl.lse_init.clone()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            ws = torch.empty(max(16, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
            plan.forward(wl.q, out, lse, ws, stream=s)
        s.synchronize()
        ref = oracle_rows(wl, prot)
        rows = [np.arange(r.q_row_begin, r.T) for r in wl.requests]
        compare(wl, out, lse, prot, ref, rows, label=f"reuse{it}")
    assert plan.device_status(stream=s) == 0


def test_lse_merge_standalone():
    """rk_lse_merge against the oracle's merge, with empty (-inf) parts and
    an all-empty pair."""
    g = torch.Generator(device="cuda").manual_seed(5)
    P, rows, H, dv = 5, 37, 3, 72
    o = torch.randn(P, rows, H, dv, device="cuda", generator=g)
    l = torch.randn(P, rows, H, device="cuda", generator=g) * 4
    l[1, :5] = float("-inf")
    l[:, 7, 1] = float("-inf")
    out = torch.empty(rows, H, dv, dtype=torch.bfloat16, device="cuda")
    lo = torch.empty(rows, H, device="cuda")
    B.lse_merge(o, l, out, lo)
    torch.cuda.synchronize()
    ro, rl = O.lse_merge(o.double().cpu().numpy(), l.double().cpu().numpy())
    go = out.double().cpu().numpy()
    gl = lo.double().cpu().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(gl), ~fin)
    assert np.abs(gl[fin] - rl[fin]).max() <= LSE_ABS
    assert np.abs(go - ro).max() <= 1e-2 * np.abs(ro).max()
    assert (go[~fin] == 0).all()
