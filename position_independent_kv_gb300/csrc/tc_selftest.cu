// Self-test of the tensor-path building blocks (test-only library).
//
// One CTA computes a single 128-row product with tcgen05.mma and writes the
// fp32 accumulator back, so the tests can compare it with a library matmul:
//   mode 0: A [128 x 64] K-major, B [128 x 64] K-major (N = 128), both
//           written to shared memory in the 128-byte swizzled layout by
//           threads;
//   mode 1: A as mode 0, B [64 x 64] stored K rows x N columns (MN-major
//           operand, N = 64);
//   mode 2: as mode 1 with A copied into tensor memory (A operand from
//           TMEM);
//   mode 3: as mode 0 with both tiles brought in by TMA tiled loads with the
//           128-byte swizzle.
// Every wait is bounded; a timeout is reported through `status`.
//
// A third check drives the kernels' bounded wait to expiry on purpose, with
// no copy and no MMA in flight (see timeout_selftest_kernel).

#include "tc_tile.cuh"

namespace rk {
namespace {

constexpr uint64_t kWaitNs = 2000000000ull;

__global__ void __launch_bounds__(128, 1)
    tc_selftest_kernel(int mode, const uint16_t* __restrict__ A, const uint16_t* __restrict__ B,
                       float* __restrict__ D, int32_t* status,
                       const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB) {
  __shared__ __align__(1024) uint8_t sA[16384];
  __shared__ __align__(1024) uint8_t sB[16384];
  __shared__ __align__(8) uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool b_mn = (mode == 1 || mode == 2);
  const int N = b_mn ? 64 : 128;

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 256);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&bar_tma, 1);
    tc::mbar_init(&bar_mma, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = tmem_base;
  bool ok = true;

  if (mode == 3) {
    if (tid == 0) {
      tc::prefetch_tmap(&tmA);
      tc::prefetch_tmap(&tmB);
      tc::mbar_arrive_expect_tx(&bar_tma, 32768);
      tc::tma_load_2d(smem_u32(sA), &tmA, &bar_tma, 0, 0);
      tc::tma_load_2d(smem_u32(sB), &tmB, &bar_tma, 0, 0);
    }
    ok = tc::mbar_wait(&bar_tma, 0, status, kWaitNs);
  } else {
    for (int i = tid; i < 128 * 64; i += 128) {
      const int r = i >> 6, c = i & 63;
      *reinterpret_cast<uint16_t*>(sA + tc::sw128_offset(r, c)) = A[i];
    }
    const int brows = b_mn ? 64 : 128;
    for (int i = tid; i < brows * 64; i += 128) {
      const int r = i >> 6, c = i & 63;
      *reinterpret_cast<uint16_t*>(sB + tc::sw128_offset(r, c)) = B[i];
    }
    tc::fence_proxy_async();
  }
  if (mode == 2) {
    // row (32 * warp + lane) of A into TMEM columns 128..159, two bf16 per column
    uint32_t r[32];
    const uint16_t* src = A + (32 * warp + lane) * 64;
#pragma unroll
    for (int c = 0; c < 32; ++c)
      r[c] = static_cast<uint32_t>(src[2 * c]) | (static_cast<uint32_t>(src[2 * c + 1]) << 16);
    tc::tmem_st32(tbase + (static_cast<uint32_t>(32 * warp) << 16) + 128, r);
    tc::tmem_wait_st();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();

  if (tid == 0 && ok) {
    const uint32_t idesc = tc::idesc_bf16(128, N, false, b_mn);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint64_t bd = b_mn ? tc::sdesc_sw128(smem_u32(sB) + 2048 * k, 1024, 1024)
                               : tc::sdesc_sw128(smem_u32(sB) + 32 * k, 16, 1024);
      if (mode == 2) {
        tc::mma_ts(tbase, tbase + 128 + 8 * k, bd, idesc, k > 0);
      } else {
        const uint64_t ad = tc::sdesc_sw128(smem_u32(sA) + 32 * k, 16, 1024);
        tc::mma_ss(tbase, ad, bd, idesc, k > 0);
      }
    }
    tc::mma_commit(&bar_mma);
  }
  if (ok) ok = tc::mbar_wait(&bar_mma, 0, status, kWaitNs);
  tc::tc_fence_after();
  if (ok) {
    for (int c = 0; c < N / 32; ++c) {
      uint32_t r[32];
      tc::tmem_ld32(tbase + (static_cast<uint32_t>(32 * warp) << 16) + 32 * c, r);
      tc::tmem_wait_ld();
      float* dst = D + (32 * warp + lane) * N + 32 * c;
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[i] = __uint_as_float(r[i]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, 256);
}

// CTA-pair check: a cluster of two CTAs computes D[256 x N] = A[256 x 64] *
// B[N x 64]^T with one tcgen05.mma.cta_group::2 per K step issued by CTA 0.
// CTA r holds rows 128r.. of A and columns (N/2)r.. of B (both K-major,
// 128-byte swizzled) and receives rows 128r.. of D in its tensor memory.
// Mode 0: N = 128 (S-shaped).  Mode 1: N = 256, B stored MN-major (K rows x
// N/2 columns per CTA, P.V-shaped).  256 columns are allocated per CTA, so
// even two separate allocations would fit in tensor memory.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    tc_2sm_selftest_kernel(int mode, const uint16_t* __restrict__ A,
                           const uint16_t* __restrict__ B, float* __restrict__ D,
                           int32_t* status, uint32_t* tmem_addr_out) {
  __shared__ __align__(1024) uint8_t sA[16384];
  __shared__ __align__(1024) uint8_t sB[16384];
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = tc::cluster_ctarank();
  const int N = mode == 1 ? 256 : 128;
  const int NH2 = N / 2;
  if (warp == 0) {
    tc::tmem_alloc_2sm(&tmem_base, 256);
    tc::tmem_relinquish_2sm();
  }
  if (tid == 0) {
    tc::mbar_init(&bar_mma, 1);
    tc::fence_barrier_init();
  }
  // this CTA's operands
  for (int i = tid; i < 128 * 64; i += 128) {
    const int r = i >> 6, c = i & 63;
    *reinterpret_cast<uint16_t*>(sA + tc::sw128_offset(r, c)) = A[(128 * rank + r) * 64 + c];
  }
  if (mode == 0) {
    for (int i = tid; i < NH2 * 64; i += 128) {
      const int r = i >> 6, c = i & 63;  // row = n within this CTA's half, col = k
      *reinterpret_cast<uint16_t*>(sB + tc::sw128_offset(r, c)) = B[(NH2 * rank + r) * 64 + c];
    }
  } else {
    // MN-major: K rows (64) x this CTA's 128 N columns as two 64-column blocks 8 KB apart
    for (int i = tid; i < 64 * NH2; i += 128) {
      const int k = i / NH2, n = i - k * NH2;
      const int blk = n >> 6, nn = n & 63;
      *reinterpret_cast<uint16_t*>(sB + blk * 8192 + tc::sw128_offset(k, nn)) =
          B[(NH2 * rank + n) * 64 + k];
    }
  }
  tc::fence_proxy_async();
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();
  tc::tc_fence_after();
  const uint32_t tbase = tmem_base;
  if (tid == 0) tmem_addr_out[rank] = tbase;
  if (rank == 0 && tid == 0) {
    const uint32_t idesc = tc::idesc_bf16(256, N, false, mode == 1);
    for (int k = 0; k < 4; ++k) {
      const uint64_t ad = tc::sdesc_sw128(smem_u32(sA) + 32 * k, 16, 1024);
      const uint64_t bd = mode == 0 ? tc::sdesc_sw128(smem_u32(sB) + 32 * k, 16, 1024)
                                    : tc::sdesc_sw128(smem_u32(sB) + 2048 * k, 8192, 1024);
      tc::mma_ss_2sm(tbase, ad, bd, idesc, k > 0);
    }
    tc::mma_commit_2sm(&bar_mma, 0x3);
  }
  const bool ok = tc::mbar_wait(&bar_mma, 0, status, kWaitNs);
  tc::tc_fence_after();
  if (ok) {
    for (int c = 0; c < N / 32; ++c) {
      uint32_t r[32];
      tc::tmem_ld32(tbase + (static_cast<uint32_t>(32 * warp) << 16) + 32 * c, r);
      tc::tmem_wait_ld();
      float* dst = D + (128 * rank + 32 * warp + lane) * N + 32 * c;
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[i] = __uint_as_float(r[i]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();
  if (warp == 0) tc::tmem_dealloc_2sm(tbase, 256);
}

// Timeout check of the kernels' bounded waits (tt::wait_bar, the wait every
// tcgen05 kernel uses).  Mode 0: no thread ever arrives on either barrier.
// Warp 0's lane 0 waits on barrier 0 with `limit_ns`; warps 2 and 3 wait on
// barrier 1 with the kernels' own 2 s bound, so they must give up as soon as
// the first waiter records the error through the CTA's abort flag, and then
// vote with bar.red.and as the softmax lanes do.  Warp 1 holds a
// tensor-memory allocation through it all and frees it at the end.  Mode 1:
// thread 0 completes both barriers first, so every wait passes.  Nothing
// else runs: no TMA copy and no MMA is in flight while a wait gives up.
// ended[0..2]: 1 if the role's wait passed, 2 if it gave up; ns[0..2]: the
// role's elapsed time.
__global__ void __launch_bounds__(128, 1)
    timeout_selftest_kernel(int mode, uint64_t limit_ns, int32_t* status, int32_t* ended,
                            unsigned long long* ns) {
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ uint32_t misc[2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    misc[1] = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(misc, 32);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = misc[0];
  if (mode == 1 && tid == 0) {
    tc::mbar_arrive(&bar[0]);
    tc::mbar_arrive(&bar[1]);
  }
  const tt::Ctx c{bar, reinterpret_cast<volatile uint32_t*>(&misc[1]), status};
  const uint64_t t0 = tc::global_ns();
  if (warp == 0) {
    if (lane == 0) {
      const bool ok = tt::wait_bar(c, 0, 0, limit_ns);
      ended[0] = ok ? 1 : 2;
      ns[0] = tc::global_ns() - t0;
    }
  } else if (warp >= 2) {
    bool ok = __all_sync(0xffffffffu, tt::wait_bar(c, 1, 0));
    ok = tc::named_and(1, 64, ok);
    if (lane == 0) {
      ended[warp - 1] = ok ? 1 : 2;
      ns[warp - 1] = tc::global_ns() - t0;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tbase, 32);
  }
}

}  // namespace
}  // namespace rk

// CTA-pair check (see above).  A: bf16 [256, 64]; B: bf16 [N, 64]; D: fp32
// [256, N]; tmem_addr_out: uint32 [2].
extern "C" int rk_tc_2sm_selftest(int mode, const void* A, const void* B, float* D,
                                  int32_t* status, uint32_t* tmem_addr_out, void* stream) {
  if (mode < 0 || mode > 1) return -1;
  rk::tc_2sm_selftest_kernel<<<2, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      mode, static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(B), D, status,
      tmem_addr_out);
  return static_cast<int>(cudaGetLastError());
}

// mode: see the file comment.  A, B: device bf16 row-major; D: device fp32
// [128, N] (N = 128 for modes 0 and 3, 64 for modes 1 and 2); status: device
// int32 (0 on entry).  Returns 0, or -1 if a tensor map cannot be encoded,
// or the CUDA error of the launch.
extern "C" int rk_tc_selftest(int mode, const void* A, const void* B, float* D, int32_t* status,
                              void* stream) {
  CUtensorMap ta{}, tb{};
  if (mode == 3) {
    const uint64_t dims[2] = {64, 128};
    const uint64_t strides[1] = {128};
    const uint32_t box[2] = {64, 128};
    if (!rk::make_tmap_bf16(&ta, A, 2, dims, strides, box)) return -1;
    if (!rk::make_tmap_bf16(&tb, B, 2, dims, strides, box)) return -1;
  }
  rk::tc_selftest_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      mode, static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(B), D, status, ta, tb);
  return static_cast<int>(cudaGetLastError());
}

// Timeout check (see above).  status: device int32 (0 on entry); ended:
// device int32 [3]; ns: device uint64 [3].  Returns 0, -1 for a bad mode or
// the launch error.
extern "C" int rk_tc_timeout_selftest(int mode, unsigned long long limit_ns, int32_t* status,
                                      int32_t* ended, unsigned long long* ns, void* stream) {
  if (mode < 0 || mode > 1) return -1;
  rk::timeout_selftest_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      mode, limit_ns, status, ended, ns);
  return static_cast<int>(cudaGetLastError());
}
