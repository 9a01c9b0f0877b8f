"""GPU parity of the rotary-value path (RK_PLAN_V_ROPE: V = the whole
latent row, each segment's output phase restored, inverse output RoPE at the
query's position; RedKnot-MLA paper, head-partition and RoPE-orthogonality
paragraphs) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle as O
from _helpers import compare, oracle_rows, run_gpu, sample_rows, untouched_all_rows
from position_independent_kv_gb300 import build as BUILD
from position_independent_kv_gb300.workloads import SPECS, make_workload

pytestmark = pytest.mark.gpu

MINI = ["flash_vrope_mini", "ctx128k_vrope_mini", "decode_vrope_mini"]


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BUILD.build()


@pytest.mark.parametrize("sharp", [False, True], ids=["stated", "sharp"])
@pytest.mark.parametrize("name", MINI)
def test_vrope_parity_every_row(name, sharp):
    """Every computed row; the sharp queries (score std ~4) make the phase of
    each segment's values decisive."""
    s = SPECS[name]
    wl = make_workload(name, seed=0, device="cuda",
                       q_scale=4.0 * (s.d_nope + s.d_rope) if sharp else 1.0)
    assert wl.v_rope and wl.d_v == 512
    out, lse, plan, bm, prot = run_gpu(wl)
    assert plan.info["d_v"] == 512
    ref = oracle_rows(wl, prot)
    rows = [np.arange(r.q_row_begin, r.T) for r in wl.requests]
    compare(wl, out, lse, prot, ref, rows, label=f"{name}/{sharp}")
    untouched_all_rows(wl, out, lse, prot)


@pytest.mark.parametrize("name", MINI)
def test_vrope_visible_key_counts_exact(name):
    """q = 0: exp(lse) counts the visible keys exactly, and the output is the
    plain mean of the visible values with their rope slices turned by
    R(k - p), compared against the oracle."""
    wl = make_workload(name, seed=0, device="cuda")
    wl.q.zero_()
    out, lse, plan, bm, prot = run_gpu(wl)
    offs = wl.row_offsets()
    glob = wl.head_role.astype(bool)
    for r, req in enumerate(wl.requests):
        p = np.arange(req.q_row_begin, req.T)
        l = lse[offs[r]:offs[r] + len(p)].double().cpu().numpy()
        cnt = np.rint(np.exp(np.minimum(l, 700.0)))
        assert np.array_equal(cnt[:, glob], np.broadcast_to((p + 1)[:, None], cnt[:, glob].shape))
    ref = oracle_rows(wl, prot)
    rows = [np.arange(r.q_row_begin, r.T) for r in wl.requests]
    compare(wl, out, lse, prot, ref, rows, label=f"{name}/q0")


def test_vrope_one_hot_phase_probe():
    """Global-head queries aimed so hard at one key k* = delta* + j* of an
    earlier segment that P is one-hot: the output is [c_nope(j*) |
    R(delta* - p) k_rope(j*)], the key's canonical rope slice moved by its
    own offset and back by the query's position (checked against that closed
    form and against the oracle)."""
    wl = make_workload("flash_vrope_mini", seed=3, device="cuda")
    req = wl.requests[0]
    rng = np.random.default_rng(5)
    glob = np.nonzero(wl.head_role)[0]
    dn = wl.d_nope
    targets = []
    for _ in range(24):
        p = int(rng.integers(300, req.T))
        cands = [s for s in req.segments if s.delta < p and not s.is_new]
        s = cands[int(rng.integers(0, len(cands)))]
        j = int(rng.integers(0, min(s.n, p - s.delta)))
        h = int(glob[int(rng.integers(0, len(glob)))])
        kn = s.latent[j, :dn].double().cpu().numpy()
        qn = kn * (40.0 / (wl.scale * float(kn @ kn)))   # ~40 nats above any other key
        wl.q[p, h] = 0
        wl.q[p, h, :dn] = torch.from_numpy(qn).to(torch.bfloat16).cuda()
        targets.append((p, h, s, j))
    out, lse, plan, bm, prot = run_gpu(wl)
    rows = [np.array(sorted({t[0] for t in targets}))]
    ref = oracle_rows(wl, prot, rows)
    compare(wl, out, lse, prot, ref, rows, label="vrope probe")
    for p, h, s, j in targets:
        lat = s.latent[j].double().cpu().numpy()
        want = np.concatenate([lat[:dn], O.rotate(lat[dn:], float(s.delta - p), wl.rope_base)])
        got = out[p, h].double().cpu().numpy()
        assert np.abs(got - want).max() <= 2e-2 * np.abs(want).max(), (p, h)


@pytest.mark.parametrize("name", ["ctx128k_vrope", "decode_vrope"])
def test_vrope_full_size_sampled(name):
    """The benchmark's rotary-value sizes in its launch configuration:
    sampled rows against the oracle, every row for the untouched bytes."""
    wl = make_workload(name, seed=0, device="cuda")
    out, lse, plan, bm, prot = run_gpu(wl)
    rng = np.random.default_rng(12)
    cap = 6 if name.startswith("decode") else 48
    rows = [sample_rows(req, prot[r], rng, wl.window, wl.sink, cap=cap)
            for r, req in enumerate(wl.requests)]
    ref = oracle_rows(wl, prot, rows)
    compare(wl, out, lse, prot, ref, rows, label=name)
    untouched_all_rows(wl, out, lse, prot)
