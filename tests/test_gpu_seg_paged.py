"""GPU parity of SegPagedAttention (RedKnot blog, "Insight 3") through the C
ABI against the fp64 oracle on the same seeded pages."""
import numpy as np
import pytest
import torch

import oracle as O
from _helpers import LSE_ABS, MAX_REL, record_stats
from position_independent_kv_gb300 import binding as B
from position_independent_kv_gb300 import build as BUILD
from position_independent_kv_gb300.paged_workloads import make_paged_workload

pytestmark = pytest.mark.gpu

# The stated bound for bf16 in / fp32 accumulate: mean relative error 2e-3,
# max error 1e-2 max|ref|, LSE 1e-3 absolute.  Two bf16 roundings set most of
# the mean error on the stated inputs: P before the P.V contraction (the
# tensor cores take V in bf16 and both operands share the type) and the
# stored output, together about 1.9e-3 here, as on the MLA path.
from _helpers import MEAN_REL  # noqa: E402

MINI = ["paged_mini", "paged_mini_g4", "paged_mini_g1", "paged_mini_g16", "paged_decode_mini",
        "paged_decode_long_mini", "paged_decode_g16_long", "paged_decode_g1_long", "paged_decode_g4", "paged_tail_g1",
        "paged_tail_g2", "paged_tail_g4_split"]


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BUILD.build()


def run(pw, flags=0):
    plan = B.SegPagedPlan.from_workload(pw, flags=flags)
    out = torch.full((pw.rows, pw.Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((pw.rows, pw.Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = None
    if plan.workspace_bytes:
        ws = torch.full((plan.workspace_bytes,), 0xA5, dtype=torch.uint8, device="cuda")
    plan.forward(pw.q, pw.k_pages, pw.v_pages, out, lse, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    return out, lse, plan


def oracle(pw, rows_per_req=None):
    kp = pw.k_pages.double().cpu().numpy()
    vp = pw.v_pages.double().cpu().numpy()
    res = []
    for r, (T, qb) in enumerate(zip(pw.seq_len, pw.q_row_begin)):
        off = pw.row_offsets()[r]
        rows = np.arange(qb, T) if rows_per_req is None else np.asarray(rows_per_req[r])
        flat = off + (rows - qb)
        q = pw.q[torch.from_numpy(flat).cuda()].double().cpu().numpy()
        bd = None if pw.block_delta is None else pw.block_delta[r]
        Oo, Lo = O.seg_paged_request(q, kp, vp, pw.block_table[r], int(T), int(qb), pw.kv_role,
                                     pw.sink, pw.window, pw.scale, 128, rows=rows, sampled=True,
                                     block_delta=bd, rope_base=pw.rope_base)
        res.append((flat, Oo, Lo))
    return res


def compare(out, lse, ref, label):
    go = np.concatenate([out[torch.from_numpy(f).cuda()].double().cpu().numpy() for f, _, _ in ref])
    gl = np.concatenate([lse[torch.from_numpy(f).cuda()].double().cpu().numpy() for f, _, _ in ref])
    ro = np.concatenate([o for _, o, _ in ref])
    rl = np.concatenate([l for _, _, l in ref])
    assert np.isfinite(go).all() and np.isfinite(gl).all(), f"{label}: unwritten or non-finite"
    err = np.abs(go - ro)
    st = dict(max_err=float(err.max()), max_ref=float(np.abs(ro).max()),
              mean_rel=float(err.sum() / np.abs(ro).sum()), lse_err=float(np.abs(gl - rl).max()),
              n=int(go.size))
    record_stats(f"seg_paged {label}", st, mean_rel=MEAN_REL)
    assert st["max_err"] <= MAX_REL * st["max_ref"], f"{label}: {st}"
    assert st["mean_rel"] <= MEAN_REL, f"{label}: {st}"
    assert st["lse_err"] <= LSE_ABS, f"{label}: {st}"
    return st


@pytest.mark.parametrize("sharp", [False, True], ids=["stated", "sharp"])
@pytest.mark.parametrize("name", MINI)
def test_seg_paged_parity_every_row(name, sharp):
    pw = make_paged_workload(name, seed=0, device="cuda", q_scale=512.0 if sharp else 1.0)
    out, lse, plan = run(pw)
    compare(out, lse, oracle(pw), f"{name}/{sharp}")


@pytest.mark.parametrize("name", ["paged_mini", "paged_mini_g4"])
def test_dense_mask_arm_same_results(name):
    """The dense + mask arm (every block, element masks) gives the same
    outputs as the paged walk, bit for bit: masked keys contribute exact
    zeros and the blocks of the paged walk come in the same order."""
    pw = make_paged_workload(name, seed=1, device="cuda", q_scale=256.0)
    o1, l1, _ = run(pw)
    o2, l2, _ = run(pw, B.RK_SEGPAGED_DENSE_MASK)
    compare(o2, l2, oracle(pw), f"{name}/dense")
    assert float((o1.float() - o2.float()).abs().max()) <= 2e-2 * float(o1.float().abs().max())


@pytest.mark.parametrize("name", MINI)
def test_seg_paged_visible_key_counts_exact(name):
    """q = 0: exp(lse) is exactly the number of visible keys of every
    (row, query head)."""
    pw = make_paged_workload(name, seed=0, device="cuda")
    pw.q.zero_()
    out, lse, plan = run(pw)
    l = lse.double().cpu().numpy()
    cnt = np.rint(np.exp(np.minimum(l, 700.0)))
    offs = pw.row_offsets()
    for r, (T, qb) in enumerate(zip(pw.seq_len, pw.q_row_begin)):
        for i, p in enumerate(range(int(qb), int(T))):
            for hq in range(pw.Hq):
                g = hq // pw.G
                want = p + 1 if pw.kv_role[g] else len(O.visible_keys(p, False, pw.sink, pw.window))
                assert cnt[offs[r] + i, hq] == want, (name, p, hq)


@pytest.mark.parametrize("name", ["qwen32b_128k", "qwen32b_decode"])
def test_seg_paged_full_size_sampled(name):
    """The benchmark sizes: sampled rows (window edges, block edges, the
    first and last rows) against the oracle."""
    pw = make_paged_workload(name, seed=0, device="cuda")
    out, lse, plan = run(pw)
    rng = np.random.default_rng(7)
    rows = []
    for T, qb in zip(pw.seq_len, pw.q_row_begin):
        T, qb = int(T), int(qb)
        if T - qb == 1:
            rows.append(np.array([qb]))
            continue
        pick = {qb, qb + 1, T - 1, 127, 128, 255, 256, 257, 383, 4095, 65535, T // 2}
        pick |= set(int(x) for x in rng.integers(qb, T, size=6))
        rows.append(np.array(sorted(x for x in pick if qb <= x < T)))
    if len(rows) > 8:  # decode: a sample of the requests, the others unchecked
        for i in range(8, len(rows)):
            rows[i] = rows[i][:0]
    ref = oracle(pw, rows)
    ref = [x for x in ref if len(x[0])]
    compare(out, lse, ref, name)
    # every computed row was written
    assert bool(torch.isfinite(lse).all()) and bool(torch.isfinite(out.float()).all())


RELOC = ["paged_reloc_mini", "paged_reloc_g8", "paged_reloc_g1", "paged_reloc_decode"]


@pytest.mark.parametrize("sharp", [False, True], ids=["stated", "sharp"])
@pytest.mark.parametrize("name", RELOC)
def test_relocated_documents_parity_every_row(name, sharp):
    """Documents cached alone and reused at other offsets (blog "Insight 1"):
    every row against the oracle, which relocates the keys physically; the
    sharp queries (score std ~4) make the relocation decisive."""
    pw = make_paged_workload(name, seed=0, device="cuda", q_scale=512.0 if sharp else 1.0)
    assert pw.block_delta is not None and (pw.block_delta != 0).any()
    out, lse, plan = run(pw)
    compare(out, lse, oracle(pw), f"{name}/reloc/{sharp}")


@pytest.mark.parametrize("name", ["paged_reloc_mini", "paged_reloc_decode"])
def test_relocated_documents_visible_key_counts_exact(name):
    pw = make_paged_workload(name, seed=0, device="cuda")
    pw.q.zero_()
    out, lse, plan = run(pw)
    cnt = np.rint(np.exp(np.minimum(lse.double().cpu().numpy(), 700.0)))
    offs = pw.row_offsets()
    for r, (T, qb) in enumerate(zip(pw.seq_len, pw.q_row_begin)):
        for i, p in enumerate(range(int(qb), int(T))):
            for hq in range(pw.Hq):
                g = hq // pw.G
                want = p + 1 if pw.kv_role[g] else len(O.visible_keys(p, False, pw.sink, pw.window))
                assert cnt[offs[r] + i, hq] == want, (name, p, hq)


def test_relocated_document_decisive_probe():
    """A query aimed at one key of a relocated document, as that key sits at
    its absolute position (R(delta) k_stored): the key must dominate the
    attention on the GPU as in the oracle, which a missing or wrong-signed
    turn of the query would not give."""
    pw = make_paged_workload("paged_reloc_mini", seed=3, device="cuda")
    r, T = 0, int(pw.seq_len[0])
    delta = pw.block_delta[r]
    blk = int(np.nonzero(delta)[0][0])          # first block of a moved document
    k_tok = blk * 128 + 5
    p = min(T - 1, k_tok + 40)
    g = int(np.nonzero(pw.kv_role)[0][0])        # a Global KV head
    page = int(pw.block_table[r, g, blk])
    kst = pw.k_pages[page, 5].double().cpu().numpy()
    th = pw.rope_base ** (-2.0 * np.arange(64) / 128)
    ang = float(delta[blk]) * th
    c, s = np.cos(ang), np.sin(ang)
    kabs = np.empty(128)
    kabs[0::2] = kst[0::2] * c - kst[1::2] * s
    kabs[1::2] = kst[0::2] * s + kst[1::2] * c
    qv = torch.from_numpy(kabs / np.linalg.norm(kabs) * 400.0).to(pw.q.dtype).cuda()
    row = int(pw.row_offsets()[r] + (p - int(pw.q_row_begin[r])))
    for h in range(g * pw.G, (g + 1) * pw.G):
        pw.q[row, h] = qv
    out, lse, plan = run(pw)
    ref = oracle(pw, [np.array([p])] + [np.zeros(0, np.int64)] * (len(pw.seq_len) - 1))
    ref = [x for x in ref if len(x[0])]
    compare(out, lse, ref, "reloc probe")
    heads = slice(g * pw.G, (g + 1) * pw.G)
    assert float(ref[0][2][0, heads].min()) > 5.0        # the probe key dominates in the oracle
    got = out[row, heads].double().cpu().numpy()
    vst = pw.v_pages[page, 5].double().cpu().numpy()
    assert np.abs(got - vst[None, :]).max() < 0.05 * np.abs(vst).max()
