// Protected-row set on the device (RedKnot-MLA paper, protected-set
// paragraph: the union of query rows Q, new rows N, dirty rows D, the first
// and last b rows of every relocated segment B_b, Indexer-selected rows
// I_top, grown by a fixed controller to a 10 / 20 / 25 % budget).
//
// One CTA per request.  A row's roles follow from the segment table alone
// (a binary search over the request's segments sorted by offset): new rows
// (RK_SEG_NEW segments) and dirty rows are always protected; cached rows are
// protected when they are boundary rows, or by the Bernoulli rule (u < p),
// or by the budget fill: the `need` non-boundary cached rows with the
// highest score (ties to the lower row), where the caller's score vector
// stands in for the Indexer.  The fill threshold is found exactly by an
// MSB-first radix select over 64-bit keys (order-preserving score bits,
// then the complemented row index, so every key is distinct).

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "rk_seg_attn.h"

namespace rk {
namespace {

constexpr int PB_THREADS = 1024;

struct PSeg {
  int64_t delta;
  int64_t n;
  int32_t is_new;
  int32_t pad;
};

struct PReq {
  int64_t T;
  int64_t seg_first;
  int64_t seg_count;
  int64_t row_first;   // offset of the request's rows in u / score / dirty
  int64_t word_first;  // offset of the request's words in the bitmaps
  int64_t need;        // rows of the budget fill (<= 0: none)
};

struct PRule {
  int64_t boundary;
  double p_random;
  int32_t mode;        // 0 boundary only, 1 Bernoulli, 2 budget, 3 none
  int32_t pad;
};

// roles of row p: bit 0 cached, bit 1 boundary, bit 2 new
__device__ __forceinline__ uint32_t row_roles(const PSeg* segs, int64_t nseg, int64_t b,
                                              int64_t p) {
  int64_t lo = 0, hi = nseg - 1;
  while (lo < hi) {  // last segment with delta <= p
    const int64_t mid = (lo + hi + 1) >> 1;
    if (segs[mid].delta <= p) lo = mid; else hi = mid - 1;
  }
  const PSeg s = segs[lo];
  const int64_t j = p - s.delta;
  if (j < 0 || j >= s.n) return 0;
  if (s.is_new) return 4u;
  const bool bnd = j < b || j >= s.n - b;
  return 1u | (bnd ? 2u : 0u);
}

__device__ __forceinline__ uint64_t fill_key(const float* score, int64_t p) {
  float f = score[p];
  uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);  // -0 ranks as +0
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(u) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(p));
}

__global__ void __launch_bounds__(PB_THREADS, 1)
    protected_build_kernel(const PReq* reqs, const PSeg* segs_all, PRule rule, const double* u,
                           const float* score, const uint32_t* dirty, uint32_t* bitmap) {
  __shared__ uint32_t hist[256];
  __shared__ uint64_t prefix_s;
  __shared__ int64_t rem_s;
  const PReq rq = reqs[blockIdx.x];
  const PSeg* segs = segs_all + rq.seg_first;
  const int tid = threadIdx.x;
  const bool fill = rule.mode == 2 && rq.need > 0;
  // ---- budget fill: the need-th largest key among the candidates ----
  uint64_t thr = ~0ull;
  if (fill) {
    if (tid == 0) {
      prefix_s = 0;
      rem_s = rq.need;
    }
    __syncthreads();
    for (int d = 7; d >= 0; --d) {
      for (int i = tid; i < 256; i += PB_THREADS) hist[i] = 0;
      __syncthreads();
      const uint64_t prefix = prefix_s;
      const uint64_t hmask = d == 7 ? 0ull : (~0ull << (8 * (d + 1)));
      for (int64_t p = tid; p < rq.T; p += PB_THREADS) {
        if ((row_roles(segs, rq.seg_count, rule.boundary, p) & 3u) != 1u) continue;
        const uint64_t k = fill_key(score + rq.row_first, p);
        if ((k & hmask) != prefix) continue;
        atomicAdd(&hist[(k >> (8 * d)) & 0xFFu], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        int64_t rem = rem_s;
        int digit = 255;
        for (; digit > 0; --digit) {
          if (static_cast<int64_t>(hist[digit]) >= rem) break;
          rem -= hist[digit];
        }
        prefix_s = prefix | (static_cast<uint64_t>(digit) << (8 * d));
        rem_s = rem;
      }
      __syncthreads();
    }
    thr = prefix_s;
  }
  // ---- bitmap words ----
  const int64_t words = (rq.T + 31) / 32;
  for (int64_t w = tid; w < words; w += PB_THREADS) {
    uint32_t bits = 0;
    for (int i = 0; i < 32; ++i) {
      const int64_t p = w * 32 + i;
      if (p >= rq.T) break;
      const uint32_t roles = row_roles(segs, rq.seg_count, rule.boundary, p);
      bool prot = (roles & 4u) != 0;
      if (dirty) prot = prot || ((dirty[rq.word_first + w] >> i) & 1u);
      if ((roles & 1u) && rule.mode != 3) {
        const bool bnd = (roles & 2u) != 0;
        if (rule.mode == 1)
          prot = prot || bnd || u[rq.row_first + p] < rule.p_random;
        else if (rule.mode == 2)
          prot = prot || bnd || (fill && fill_key(score + rq.row_first, p) >= thr);
        else
          prot = prot || bnd;
      }
      bits |= (prot ? 1u : 0u) << i;
    }
    bitmap[rq.word_first + w] = bits;
  }
}

}  // namespace
}  // namespace rk

extern "C" size_t rk_protected_workspace_bytes(int32_t num_requests, int32_t num_segments) {
  if (num_requests < 1 || num_segments < 1) return 0;
  const size_t a = (static_cast<size_t>(num_requests) * sizeof(rk::PReq) + 255) & ~size_t(255);
  return a + static_cast<size_t>(num_segments) * sizeof(rk::PSeg);
}

extern "C" rk_status_t rk_protected_build(int32_t num_requests, const int32_t* seg_begin,
                                          const rk_segment_t* segs, int32_t boundary,
                                          double p_random, int32_t budget_pct, uint32_t rule_flags,
                                          const double* u, const float* score,
                                          const uint32_t* dirty, uint32_t* bitmap,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  using rk::PReq;
  using rk::PSeg;
  if (!seg_begin || !segs || !bitmap || !workspace) return RK_ERR_NULL;
  if (num_requests < 1 || boundary < 0 || budget_pct < 0 || budget_pct > 100 ||
      !(p_random >= 0.0 && p_random <= 1.0) || (rule_flags & ~RK_PROT_NONE))
    return RK_ERR_INVALID_ARG;
  if (seg_begin[0] != 0) return RK_ERR_INVALID_ARG;
  for (int r = 0; r < num_requests; ++r)
    if (seg_begin[r + 1] <= seg_begin[r]) return RK_ERR_INVALID_ARG;
  const int32_t nseg = seg_begin[num_requests];
  if (workspace_bytes < rk_protected_workspace_bytes(num_requests, nseg)) return RK_ERR_WORKSPACE;
  rk::PRule rule{};
  rule.boundary = boundary;
  rule.p_random = p_random;
  rule.mode = (rule_flags & RK_PROT_NONE) ? 3 : (p_random > 0.0 ? 1 : (budget_pct > 0 ? 2 : 0));
  if (rule.mode == 1 && !u) return RK_ERR_NULL;
  if (rule.mode == 2 && !score) return RK_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(bitmap) | reinterpret_cast<uintptr_t>(dirty)) & 3)
    return RK_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(workspace) & 15) return RK_ERR_ALIGNMENT;

  std::vector<PReq> reqs(num_requests);
  std::vector<PSeg> ps(nseg);
  int64_t row_off = 0, word_off = 0;
  for (int r = 0; r < num_requests; ++r) {
    const int b = seg_begin[r], e = seg_begin[r + 1];
    std::vector<int> idx(e - b);
    for (int j = 0; j < e - b; ++j) idx[j] = b + j;
    std::stable_sort(idx.begin(), idx.end(),
                     [&](int x, int y) { return segs[x].delta < segs[y].delta; });
    int64_t pos = 0, C = 0, B = 0;
    for (int j = 0; j < e - b; ++j) {
      const rk_segment_t& s = segs[idx[j]];
      if (s.n < 1 || s.delta < 0 || (s.flags & ~RK_SEG_NEW)) return RK_ERR_INVALID_ARG;
      if (s.delta < pos) return RK_ERR_SEGMENT_OVERLAP;
      if (s.delta > pos) return RK_ERR_SEGMENT_GAP;
      pos = s.delta + s.n;
      if (pos > INT32_MAX) return RK_ERR_CAPACITY;
      PSeg& d = ps[b + j];
      d.delta = s.delta;
      d.n = s.n;
      d.is_new = (s.flags & RK_SEG_NEW) ? 1 : 0;
      d.pad = 0;
      if (!d.is_new) {
        C += s.n;
        B += std::min<int64_t>(s.n, 2 * static_cast<int64_t>(boundary));
      }
    }
    PReq& q = reqs[r];
    q.T = pos;
    q.seg_first = b;
    q.seg_count = e - b;
    q.row_first = row_off;
    q.word_first = word_off;
    // budget target ceil(pct * C / 100) over the cached rows, boundary rows first
    q.need = rule.mode == 2 ? (static_cast<int64_t>(budget_pct) * C + 99) / 100 - B : 0;
    row_off += pos;
    word_off += (pos + 31) / 32;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(workspace);
  const size_t a = (static_cast<size_t>(num_requests) * sizeof(PReq) + 255) & ~size_t(255);
  PReq* d_reqs = reinterpret_cast<PReq*>(w);
  PSeg* d_segs = reinterpret_cast<PSeg*>(w + a);
  // the host tables are pageable: these copies are staged before returning
  if (cudaMemcpyAsync(d_reqs, reqs.data(), reqs.size() * sizeof(PReq), cudaMemcpyHostToDevice, s) !=
          cudaSuccess ||
      cudaMemcpyAsync(d_segs, ps.data(), ps.size() * sizeof(PSeg), cudaMemcpyHostToDevice, s) !=
          cudaSuccess)
    return RK_ERR_CUDA;
  rk::protected_build_kernel<<<num_requests, rk::PB_THREADS, 0, s>>>(d_reqs, d_segs, rule, u,
                                                                      score, dirty, bitmap);
  return cudaGetLastError() == cudaSuccess ? RK_OK : RK_ERR_CUDA;
}
