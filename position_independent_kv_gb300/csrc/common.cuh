// Device helpers shared by the kernels: bf16 packing, ldmatrix, mma.sync,
// cp.async and the fast exp2 instruction.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "rk_internal.h"

namespace rk {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t x) {
  return __uint_as_float(static_cast<uint32_t>(x) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&b);
}

// 2^x with the hardware approximation (flush-to-zero); exp2(-inf) = 0.
// Not volatile: the compiler may schedule it like any arithmetic.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
      "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 16-byte asynchronous global->shared copy; bytes beyond src_bytes are zero.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Next key tile of a work item.  Keys visited: [r0lo, r0hi) u [r1lo, r1hi)
// intersected with each segment (segments sorted by offset), walked segment
// by segment so the query rotation changes only at segment boundaries.
// `skip` (from the plan, 0 = none) names segments [skip & 0xffff, skip >> 16)
// that meet neither range: the walk jumps over them instead of reading each
// one's offset, which between a sink and a window far behind it would be a
// chain of dependent global loads.
struct KeyTile {
  int j;    // segment index within the request
  int rr;   // range 0 (sink) or 1 (window / causal)
  int k0;   // absolute first key
  int k1;   // absolute end key (exclusive); -1 before the first tile
};

template <int TN>
__device__ __forceinline__ bool next_key_tile(KeyTile& t, const DevSeg* segs, int nseg, int r0lo,
                                              int r0hi, int r1lo, int r1hi,
                                              uint32_t skip = 0) {
  const int jlo = static_cast<int>(skip & 0xffffu), jhi = static_cast<int>(skip >> 16);
  int j = t.j, rr = t.rr, k = t.k1;
  while (j < nseg) {
    const int d = segs[j].delta;
    const int e = d + segs[j].n;
    const int lo = max(rr ? r1lo : r0lo, d);
    const int hi = min(rr ? r1hi : r0hi, e);
    const int start = (k < 0) ? lo : max(k, lo);
    if (start < hi) {
      t.j = j;
      t.rr = rr;
      t.k0 = start;
      t.k1 = min(start + TN, hi);
      return true;
    }
    if (rr == 0) {
      rr = 1;
    } else {
      rr = 0;
      ++j;
      if (j >= jlo && j < jhi) j = jhi;
    }
    k = -1;
  }
  return false;
}

}  // namespace rk
