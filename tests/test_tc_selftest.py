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


def test_data_movement_probes(selftest_lib):
    """Hardware probes behind the prefill kernels' data movement (run with -s
    to see the tables): TMA streaming throughput over all SMs by box shape for
    per-CTA loads, CTA-pair loads completing on the leader's barrier, and
    per-CTA loads whose arrival is forwarded to the leader; then the round trip
    of remote mbarrier arrives between the CTAs of a pair.  Asserts only that
    every probe runs to completion without an expired wait."""
    L = selftest_lib
    L.rk_tma_stream_probe.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 6 + [ctypes.c_void_p] * 2
    L.rk_tma_stream_probe.restype = ctypes.c_int
    L.rk_tma_pair_probe.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 7 + [ctypes.c_void_p] * 2
    L.rk_tma_pair_probe.restype = ctypes.c_int
    L.rk_remote_arrive_probe.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p] * 3
    L.rk_remote_arrive_probe.restype = ctypes.c_int
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ctas = sms - (sms & 1)
    rows = 131072
    g = torch.Generator(device="cuda").manual_seed(7)
    lat = torch.randn(rows, 576, device="cuda", generator=g).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    clk = 2.07e9  # the part's maximum SM clock, for B/clk/SM
    print(f"\nTMA streaming, {ctas} CTAs, [{rows}, 576] bf16, box 64 dims x rows x chunks")
    print("box           bytes  slots  per-CTA  pair  forwarded   (B/clk/SM)")
    for br, bc, slots in [(64, 3, 5), (128, 2, 4), (64, 4, 3), (64, 9, 2), (128, 4, 3)]:
        bb = 128 * br * bc
        n = max(16, int(24e6 // bb))
        res = []
        for mode in (0, 1, 2):
            best = None
            for _ in range(2):
                e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
                e0.record()
                rc = L.rk_tma_pair_probe(lat.data_ptr(), rows, br, bc, slots, n, mode, ctas,
                                         status.data_ptr(), stream)
                e1.record()
                torch.cuda.synchronize()
                assert rc == 0
                ms = e0.elapsed_time(e1)
                best = ms if best is None else min(best, ms)
            assert int(status.item()) == 0, "a bounded wait expired"
            res.append(ctas * n * bb / (best * 1e-3) / ctas / clk)
        print(f"{br:3d} x {bc}     {bb // 1024:3d} KB  {slots:4d}  {res[0]:7.1f} {res[1]:5.1f} {res[2]:8.1f}")
    ns = torch.zeros(1, dtype=torch.int64, device="cuda")
    for relaxed in (0, 1):
        n = 20000
        assert L.rk_remote_arrive_probe(n, relaxed, ctas, status.data_ptr(), ns.data_ptr(),
                                        stream) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0, "a bounded wait expired"
        print(f"remote mbarrier arrive round trip ({'relaxed' if relaxed else 'release'}): "
              f"{int(ns.item()) / n:.1f} ns")
