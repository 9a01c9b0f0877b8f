"""Tensor-path building blocks on the GPU: tcgen05.mma with 128-byte
swizzled shared-memory descriptors (K-major and MN-major B), A from tensor
memory, and TMA tiled loads, each checked against a float64 matmul."""
import ctypes

import pytest
import torch

from position_independent_kv_gb300 import build as BUILD

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def selftest_lib():
    assert torch.cuda.is_available()
    BUILD.build()
    L = ctypes.CDLL(BUILD.SELFTEST_LIB)
    L.rk_tc_selftest.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                 ctypes.c_void_p, ctypes.c_void_p]
    L.rk_tc_selftest.restype = ctypes.c_int
    return L


@pytest.mark.parametrize("mode", [0, 1, 2, 3],
                         ids=["ss_kmajor", "ss_b_mnmajor", "ts_b_mnmajor", "tma_ss_kmajor"])
def test_tcgen05_building_blocks(selftest_lib, mode):
    g = torch.Generator(device="cuda").manual_seed(100 + mode)
    A = torch.randn(128, 64, device="cuda", generator=g).to(torch.bfloat16)
    if mode in (1, 2):
        B = torch.randn(64, 64, device="cuda", generator=g).to(torch.bfloat16)
        ref = A.double().cpu() @ B.double().cpu()
    else:
        B = torch.randn(128, 64, device="cuda", generator=g).to(torch.bfloat16)
        ref = A.double().cpu() @ B.double().cpu().T
    D = torch.full(tuple(ref.shape), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = selftest_lib.rk_tc_selftest(mode, A.data_ptr(), B.data_ptr(), D.data_ptr(),
                                     status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert int(status.item()) == 0, "a bounded wait expired"
    got = D.double().cpu()
    err = (got - ref).abs()
    assert torch.isfinite(got).all(), "accumulator not fully written"
    assert float(err.max()) <= 1e-3 * max(1.0, float(ref.abs().max())), (
        f"mode {mode}: max err {float(err.max())}, first row got {got[0, :6].tolist()} "
        f"want {ref[0, :6].tolist()}")


@pytest.mark.parametrize("mode", [0, 1], ids=["pair_n128_kmajor", "pair_n256_mnmajor"])
def test_tcgen05_cta_pair(selftest_lib, mode):
    """tcgen05.mma.cta_group::2 over a cluster of two CTAs: A and D rows
    split between the CTAs, B split along N, one issuing thread, completion
    multicast to both CTAs."""
    L = selftest_lib
    L.rk_tc_2sm_selftest.argtypes = [ctypes.c_int] + [ctypes.c_void_p] * 6
    L.rk_tc_2sm_selftest.restype = ctypes.c_int
    N = 256 if mode == 1 else 128
    g = torch.Generator(device="cuda").manual_seed(200 + mode)
    A = torch.randn(256, 64, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, 64, device="cuda", generator=g).to(torch.bfloat16)
    D = torch.full((256, N), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    taddr = torch.full((2,), 0xFFFFFFFF, dtype=torch.int64, device="cuda").to(torch.int32)
    rc = L.rk_tc_2sm_selftest(mode, A.data_ptr(), B.data_ptr(), D.data_ptr(), status.data_ptr(),
                              taddr.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert int(status.item()) == 0, "a bounded wait expired"
    t = taddr.cpu().tolist()
    assert t[0] == t[1], f"the pair got different TMEM addresses {t}"
    ref = A.double().cpu() @ B.double().cpu().T
    got = D.double().cpu()
    assert torch.isfinite(got).all(), "accumulator not fully written"
    err = (got - ref).abs()
    assert float(err.max()) <= 1e-3 * max(1.0, float(ref.abs().max())), (
        f"mode {mode}: max err {float(err.max())}; row 0 {got[0, :4].tolist()} vs "
        f"{ref[0, :4].tolist()}; row 128 {got[128, :4].tolist()} vs {ref[128, :4].tolist()}")


def test_bounded_wait_expires_cleanly(selftest_lib):
    """The kernels' bounded wait run out on purpose, with no copy and no MMA
    in flight: a waiter on a barrier that nothing completes gives up after
    its limit and records RK_ERR_DEVICE_TIMEOUT (8); the CTA's other roles,
    waiting with the kernels' own 2 s bound, give up at once through the
    abort flag and leave their bar.red vote together; tensor memory is freed;
    the launch returns.  The context stays usable: a following forward
    through the C ABI matches the oracle and reports a clean status."""
    import numpy as np
    from _helpers import compare, oracle_rows, run_gpu
    from position_independent_kv_gb300.workloads import make_workload
    L = selftest_lib
    L.rk_tc_timeout_selftest.argtypes = [ctypes.c_int, ctypes.c_ulonglong] + [ctypes.c_void_p] * 4
    L.rk_tc_timeout_selftest.restype = ctypes.c_int
    stream = torch.cuda.current_stream().cuda_stream

    def run(mode, limit_ns):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        ended = torch.zeros(3, dtype=torch.int32, device="cuda")
        ns = torch.zeros(3, dtype=torch.int64, device="cuda")
        e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
        e0.record()
        rc = L.rk_tc_timeout_selftest(mode, limit_ns, status.data_ptr(), ended.data_ptr(),
                                      ns.data_ptr(), stream)
        e1.record()
        torch.cuda.synchronize()
        assert rc == 0
        return int(status.item()), ended.tolist(), ns.tolist(), e0.elapsed_time(e1)

    # every barrier completed: every wait passes, no error
    st, ended, ns, _ = run(1, 20_000)
    assert st == 0 and ended == [1, 1, 1], (st, ended)
    # nothing completes barrier 0: its waiter gives up after 20 us, the other
    # roles follow it long before their own 2 s bound
    limit = 20_000
    st, ended, ns, ms = run(0, limit)
    assert st == 8, f"status {st}, want RK_ERR_DEVICE_TIMEOUT"
    assert ended == [2, 2, 2], ended
    assert ns[0] >= limit, ns
    assert max(ns) < 100_000_000, f"a role kept waiting after the abort: {ns} ns"
    assert ms < 1000.0
    print(f"\nbounded wait: first waiter gave up after {ns[0] / 1e3:.1f} us, "
          f"the others after {ns[1] / 1e3:.1f} / {ns[2] / 1e3:.1f} us; launch {ms:.3f} ms")
    # the context is intact: a normal forward is correct and its status clean
    wl = make_workload("tiny", seed=0, device="cuda")
    out, lse, plan, bm, prot = run_gpu(wl)
    ref = oracle_rows(wl, prot)
    rows = [np.arange(r.q_row_begin, r.T) for r in wl.requests]
    compare(wl, out, lse, prot, ref, rows, label="tiny after an expired wait")
