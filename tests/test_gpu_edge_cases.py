"""GPU parity on the degenerate cases of the method, every computed row
against the fp64 oracle, on the default 4-CTA kernel and the CTA-pair
kernel (the mma.sync kernel where the tensor-memory kernels do not apply):
no sink and a zero window (a Local row sees only itself), one-row segments,
decode requests of one to ten rows, the smallest head count (H = 8), and
forty segments of one to nine rows with one row per Local tile."""
import numpy as np
import pytest
import torch

import oracle as O
from _helpers import compare, oracle_rows, run_gpu, untouched_all_rows
from position_independent_kv_gb300 import binding as B
from position_independent_kv_gb300 import build as BUILD
from position_independent_kv_gb300.workloads import SPECS, make_workload

pytestmark = pytest.mark.gpu

EDGE = ["edge_sink0_w0", "edge_tiny_decode", "edge_h8", "edge_many_segs"]


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BUILD.build()


@pytest.mark.parametrize("flags", [0, B.RK_PLAN_CTA_PAIR], ids=["default", "cta_pair"])
@pytest.mark.parametrize("sharp", [False, True], ids=["stated", "sharp"])
@pytest.mark.parametrize("name", EDGE)
def test_edge_parity_every_row(name, sharp, flags):
    s = SPECS[name]
    wl = make_workload(name, seed=0, device="cuda", q_scale=4.0 * (s.d_nope + s.d_rope) if sharp else 1.0)
    out, lse, plan, bm, prot = run_gpu(wl, flags=flags)
    ref = oracle_rows(wl, prot)
    rows = [np.arange(r.q_row_begin, r.T) for r in wl.requests]
    compare(wl, out, lse, prot, ref, rows, label=f"{name}/{flags}/{sharp}")
    untouched_all_rows(wl, out, lse, prot)


@pytest.mark.parametrize("name", EDGE)
def test_edge_key_counts_exact(name):
    """q = 0: exp(lse) equals the number of visible keys of every computed
    (row, head) pair, including the one-key rows of a zero window."""
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
        new = np.zeros(req.T, bool)
        for sg in req.segments:
            if sg.is_new:
                new[sg.delta:sg.delta + sg.n] = True
        pr = (prot[r] | new)[req.q_row_begin:]
        if (~glob).any() and pr.any():
            want = np.array([len(O.visible_keys(int(x), False, wl.sink, wl.window)) for x in p[pr]],
                            dtype=np.float64)
            assert np.array_equal(cnt[pr][:, ~glob], np.broadcast_to(want[:, None], cnt[pr][:, ~glob].shape))
