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

// Streaming probe: each CTA pulls `chunks` boxes of 64 bf16 x box_rows rows
// of a [rows, 576] bf16 tensor through a ring of `slots` shared-memory
// buffers; one thread issues the TMA loads, another releases each buffer as
// soon as it lands.  Measures how much data a ring depth keeps in flight.
__global__ void __launch_bounds__(64, 1)
    tma_stream_probe_kernel(const __grid_constant__ CUtensorMap tm, int rows, int box_rows,
                            int box_chunks, int slots, int chunks, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t box_bytes = 128u * box_rows * box_chunks;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + slots * box_bytes);
  uint64_t* empty = full + slots;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < slots; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    tc::fence_barrier_init();
  }
  __syncthreads();
  const int span = rows - box_rows;
  if (tid == 0) {
    for (int c = 0; c < chunks; ++c) {
      const int slot = c % slots;
      const uint32_t ph = (c / slots) & 1;
      if (!tc::mbar_wait(&empty[slot], ph ^ 1, status, kWaitNs)) return;
      tc::mbar_arrive_expect_tx(&full[slot], box_bytes);
      const int t = blockIdx.x * chunks + c;
      const int y = static_cast<int>((static_cast<int64_t>(t / 9) * box_rows) % span);
      if (box_chunks == 1)
        tc::tma_load_2d(smem_u32(sm + slot * box_bytes), &tm, &full[slot], 64 * (t % 9), y);
      else
        tc::tma_load_3d(smem_u32(sm + slot * box_bytes), &tm, &full[slot], 0, y,
                        (t % (10 - box_chunks)));
    }
    for (int c = chunks > slots ? chunks - slots : 0; c < chunks; ++c)
      tc::mbar_wait(&full[c % slots], (c / slots) & 1, status, kWaitNs);
  } else if (tid == 32) {
    for (int c = 0; c < chunks; ++c) {
      const int slot = c % slots;
      if (!tc::mbar_wait(&full[slot], (c / slots) & 1, status, kWaitNs)) return;
      tc::mbar_arrive(&empty[slot]);
    }
  }
}

// MMA rate probe: one CTA issues `iters` MMAs of one shape back to back on
// resident operands and reports the elapsed nanoseconds from the first issue
// to the completion of the last (mode 0: SS, M=128 N=128 K=16, both K-major;
// mode 1: TS, M=128 N=64, A from TMEM, B MN-major; mode 2: SS M=128 N=256).
__global__ void __launch_bounds__(128, 1)
    tc_rate_kernel(int mode, int iters, unsigned long long* ns, int32_t* status) {
  extern __shared__ uint8_t dyn[];
  uint8_t* sA = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sB = sA + 16384;
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < 16384 / 4; i += 128) reinterpret_cast<uint32_t*>(sA)[i] = 0x3f803f80u;
  for (int i = tid; i < 32768 / 4; i += 128) reinterpret_cast<uint32_t*>(sB)[i] = 0x3f803f80u;
  tc::fence_proxy_async();
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&bar_mma, 1);
    tc::fence_barrier_init();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = tmem_base;
  if (tid == 0) {
    const int N = mode == 1 ? 64 : (mode == 2 ? 256 : 128);
    const uint32_t idesc = tc::idesc_bf16(128, N, false, mode == 1);
    const uint64_t ad = tc::sdesc_sw128(smem_u32(sA), 16, 1024);
    const uint64_t bd = mode == 1 ? tc::sdesc_sw128(smem_u32(sB), 1024, 1024)
                                  : tc::sdesc_sw128(smem_u32(sB), 16, 1024);
    const uint64_t t0 = tc::global_ns();
    for (int i = 0; i < iters; ++i) {
      if (mode == 1)
        tc::mma_ts(tbase, tbase + 256, bd, idesc, i > 0);
      else
        tc::mma_ss(tbase, ad, bd, idesc, i > 0);
    }
    tc::mma_commit(&bar_mma);
    tc::mbar_wait(&bar_mma, 0, status, kWaitNs);
    ns[0] = tc::global_ns() - t0;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, 512);
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


// Pair streaming probe: clusters of two CTAs pull `n` boxes each of a
// [rows, 576] bf16 tensor (viewed (64, rows, 9), box 64 x box_rows x
// box_chunks) through `slots` buffers.  mode 0: each CTA loads into its own
// buffer on its own barrier and releases it on arrival; mode 1: both CTAs'
// boxes complete on rank 0's barrier (cta_group::2 form) and rank 0 releases
// the slot in both CTAs; mode 2: each CTA loads on its own barrier, rank 1
// forwards its arrival to rank 0 with a remote arrive, and rank 0 releases
// the slot in both CTAs.  Every wait is bounded.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(64, 1)
    tma_pair_probe_kernel(const __grid_constant__ CUtensorMap tm, int rows, int box_rows,
                          int box_chunks, int slots, int n, int mode, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t bb = 128u * box_rows * box_chunks;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + slots * bb);
  uint64_t* empty = full + slots;
  uint64_t* peer = empty + slots;
  const int tid = threadIdx.x;
  const uint32_t rank = tc::cluster_ctarank();
  if (tid == 0) {
    for (int i = 0; i < slots; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
      tc::mbar_init(&peer[i], 1);
    }
    tc::fence_barrier_init();
  }
  __syncthreads();
  tc::cluster_sync();
  const int span = rows - box_rows;
  if (tid == 0) {
    for (int c = 0; c < n; ++c) {
      const int slot = c % slots;
      if (!tc::mbar_wait(&empty[slot], ((c / slots) & 1) ^ 1, status, kWaitNs)) break;
      const int y = (c * box_rows + 64 * static_cast<int>(rank)) % span;
      if (mode == 1) {
        if (rank == 0) tc::mbar_arrive_expect_tx(&full[slot], 2 * bb);
        tc::tma_load_3d_2sm(smem_u32(sm + slot * bb), &tm,
                            tc::mapa_shared(smem_u32(&full[slot]), 0), 0, y, 0);
      } else {
        tc::mbar_arrive_expect_tx(&full[slot], bb);
        tc::tma_load_3d(smem_u32(sm + slot * bb), &tm, &full[slot], 0, y, 0);
      }
    }
    // copies in flight land before the CTA exits
    for (int c = n > slots ? n - slots : 0; c < n && (mode != 1 || rank == 0); ++c)
      tc::mbar_wait(&full[c % slots], (c / slots) & 1, status, kWaitNs);
  } else if (tid == 32) {
    for (int c = 0; c < n; ++c) {
      const int slot = c % slots;
      const uint32_t ph = (c / slots) & 1;
      if (mode == 0) {
        if (!tc::mbar_wait(&full[slot], ph, status, kWaitNs)) break;
        tc::mbar_arrive(&empty[slot]);
      } else if (rank == 1) {
        if (mode == 2) {
          if (!tc::mbar_wait(&full[slot], ph, status, kWaitNs)) break;
          tc::mbar_arrive_cluster(tc::mapa_shared(smem_u32(&peer[slot]), 0));
        }
      } else {
        if (!tc::mbar_wait(&full[slot], ph, status, kWaitNs)) break;
        if (mode == 2 && !tc::mbar_wait(&peer[slot], ph, status, kWaitNs)) break;
        tc::mbar_arrive(&empty[slot]);
        tc::mbar_arrive_cluster(tc::mapa_shared(smem_u32(&empty[slot]), 1));
      }
    }
  }
  __syncthreads();
  tc::cluster_sync();
}

// Remote-arrive ping-pong between the two CTAs of a cluster: `n` round trips
// of one arrive each way (release or relaxed at cluster scope); rank 0 of
// cluster 0 reports the elapsed nanoseconds.
__global__ void __cluster_dims__(2, 1, 1)
    remote_arrive_probe_kernel(int n, int relaxed, int32_t* status, unsigned long long* ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t rank = tc::cluster_ctarank();
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  tc::cluster_sync();
  const uint32_t other = tc::mapa_shared(smem_u32(&bar), rank ^ 1);
  auto arrive = [&]() {
    if (relaxed)
      asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(other)
                   : "memory");
    else
      tc::mbar_arrive_cluster(other);
  };
  const uint64_t t0 = tc::global_ns();
  if (threadIdx.x == 0) {
    for (int i = 0; i < n; ++i) {
      if (rank == 0) {
        arrive();
        if (!tc::mbar_wait(&bar, i & 1, status, kWaitNs)) break;
      } else {
        if (!tc::mbar_wait(&bar, i & 1, status, kWaitNs)) break;
        arrive();
      }
    }
  }
  __syncthreads();
  tc::cluster_sync();
  if (threadIdx.x == 0 && rank == 0 && blockIdx.x == 0) ns[0] = tc::global_ns() - t0;
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

extern "C" int rk_tc_mma_rate(int mode, int iters, unsigned long long* ns, int32_t* status,
                              void* stream) {
  if (mode < 0 || mode > 2 || iters < 1) return -1;
  const int smem = 16384 + 32768 + 1024;
  cudaError_t e = cudaFuncSetAttribute(rk::tc_rate_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return static_cast<int>(e);
  rk::tc_rate_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(mode, iters, ns, status);
  return static_cast<int>(cudaGetLastError());
}

// TMA streaming probe (see above).  lat: device bf16 [rows, 576].  Returns 0
// or -1 (bad arguments / tensor map) or the launch error.
extern "C" int rk_tma_stream_probe(const void* lat, int rows, int box_rows, int box_chunks,
                                   int slots, int chunks, int ctas, int32_t* status,
                                   void* stream) {
  if (box_rows < 8 || box_rows > 256 || slots < 1 || slots > 13 || rows <= box_rows) return -1;
  if (box_chunks < 1 || box_chunks > 9) return -1;
  const int64_t bb = static_cast<int64_t>(128) * box_rows * box_chunks;
  if (slots * bb > 200 * 1024) return -1;
  CUtensorMap tm{};
  if (box_chunks == 1) {
    const uint64_t dims[2] = {576, static_cast<uint64_t>(rows)};
    const uint64_t strides[1] = {1152};
    const uint32_t box[2] = {64, static_cast<uint32_t>(box_rows)};
    if (!rk::make_tmap_bf16(&tm, lat, 2, dims, strides, box)) return -1;
  } else {
    // the row viewed as 9 chunks of 64: dims (64, rows, 9), the box lands
    // chunk-major in shared memory
    const uint64_t dims[3] = {64, static_cast<uint64_t>(rows), 9};
    const uint64_t strides[2] = {1152, 128};
    const uint32_t box[3] = {64, static_cast<uint32_t>(box_rows), static_cast<uint32_t>(box_chunks)};
    if (!rk::make_tmap_bf16(&tm, lat, 3, dims, strides, box)) return -2;
  }
  const size_t smem = static_cast<size_t>(slots * bb) + 2 * 13 * 8 + 1024;
  cudaError_t e = cudaFuncSetAttribute(rk::tma_stream_probe_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return static_cast<int>(e);
  rk::tma_stream_probe_kernel<<<ctas, 64, smem, static_cast<cudaStream_t>(stream)>>>(
      tm, rows, box_rows, box_chunks, slots, chunks, status);
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

// Pair streaming probe (see above): ctas (even) CTAs in clusters of two.
// lat: device bf16 [rows, 576].  Returns 0, -1 (bad arguments or tensor map)
// or the launch error.
extern "C" int rk_tma_pair_probe(const void* lat, int rows, int box_rows, int box_chunks,
                                 int slots, int n, int mode, int ctas, int32_t* status,
                                 void* stream) {
  if (box_rows < 8 || box_rows > 256 || box_chunks < 1 || box_chunks > 9 || slots < 1 ||
      slots > 8 || rows <= box_rows + 64 || n < 1 || mode < 0 || mode > 2 || ctas < 2 ||
      (ctas & 1))
    return -1;
  const int64_t bb = static_cast<int64_t>(128) * box_rows * box_chunks;
  if (slots * bb > 200 * 1024) return -1;
  CUtensorMap tm{};
  const uint64_t dims[3] = {64, static_cast<uint64_t>(rows), 9};
  const uint64_t strides[2] = {1152, 128};
  const uint32_t box[3] = {64, static_cast<uint32_t>(box_rows), static_cast<uint32_t>(box_chunks)};
  if (!rk::make_tmap_bf16(&tm, lat, 3, dims, strides, box)) return -1;
  const size_t smem = static_cast<size_t>(slots * bb) + 3 * 8 * 8 + 1024;
  cudaError_t e = cudaFuncSetAttribute(rk::tma_pair_probe_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return static_cast<int>(e);
  rk::tma_pair_probe_kernel<<<ctas, 64, smem, static_cast<cudaStream_t>(stream)>>>(
      tm, rows, box_rows, box_chunks, slots, n, mode, status);
  return static_cast<int>(cudaGetLastError());
}

// Remote-arrive ping-pong (see above) on `ctas` (even) CTAs.
extern "C" int rk_remote_arrive_probe(int n, int relaxed, int ctas, int32_t* status,
                                      unsigned long long* ns, void* stream) {
  if (n < 1 || ctas < 2 || (ctas & 1)) return -1;
  rk::remote_arrive_probe_kernel<<<ctas, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      n, relaxed, status, ns);
  return static_cast<int>(cudaGetLastError());
}
