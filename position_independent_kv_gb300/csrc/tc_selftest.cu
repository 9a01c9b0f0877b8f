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

#include "tc_ptx.cuh"
#include "tmap.h"

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

}  // namespace
}  // namespace rk

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
