// Pieces shared by the tcgen05 prefill-tile kernels: bounded mbarrier waits,
// the (row, head) of a tile lane, the rotated q_rope written to tensor
// memory, and the TMA maps and loads of a tile's queries.
#pragma once

#include "tc_ptx.cuh"
#include "tmap.h"

namespace rk {
namespace tt {

constexpr uint64_t WAIT_NS = 2000000000ull;  // bound of every wait: 2 s

struct Ctx {
  uint64_t* bar;              // this CTA's barrier array
  volatile uint32_t* abort;   // set by any role of this CTA that gives up
  int32_t* status;            // the launch's device status word
};

// Bounded wait for the phase with `parity` of barrier i; also gives up as
// soon as another role of this CTA, or any CTA of the launch, has recorded
// an error.  On expiry records RK_ERR_DEVICE_TIMEOUT.
// CLUSTER: the phase is completed by arrivals from other CTAs that publish
// shared-memory data: relaxed polls at cluster scope, then a shared-memory
// acquire fence at cluster scope.
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_bar(const Ctx& c, int i, uint32_t parity,
                                         uint64_t limit_ns = WAIT_NS) {
  uint64_t* b = c.bar + i;
  uint32_t it = 0;
  uint64_t t0 = 0;
  while (!(CLUSTER ? tc::mbar_try_wait_cluster(b, parity) : tc::mbar_try_wait(b, parity))) {
    if ((++it & 63u) == 0) {
      if (*c.abort || *reinterpret_cast<volatile int32_t*>(c.status)) {
        *c.abort = 1;
        return false;
      }
      const uint64_t now = tc::global_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit_ns) {
        *c.abort = 1;
        atomicCAS(c.status, 0, static_cast<int32_t>(RK_ERR_DEVICE_TIMEOUT));
        return false;
      }
    }
  }
  if (CLUSTER) tc::fence_acquire_cluster_smem();
  return true;
}

// Bounded wait until the monotonic counter `cnt` (in this CTA's shared
// memory, written by release stores from other CTAs of the cluster) reaches
// `need`, polled with relaxed loads and closed by a shared-memory acquire
// fence; the same give-up rules as wait_bar.
__device__ __forceinline__ bool wait_count(const Ctx& c, const uint32_t* cnt, uint32_t need,
                                           uint64_t limit_ns = WAIT_NS) {
  uint32_t it = 0;
  uint64_t t0 = 0;
  while (tc::ld_relaxed_cluster_u32(cnt) < need) {
    if ((++it & 63u) == 0) {
      if (*c.abort || *reinterpret_cast<volatile int32_t*>(c.status)) {
        *c.abort = 1;
        return false;
      }
      const uint64_t now = tc::global_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit_ns) {
        *c.abort = 1;
        atomicCAS(c.status, 0, static_cast<int32_t>(RK_ERR_DEVICE_TIMEOUT));
        return false;
      }
    }
  }
  tc::fence_acquire_cluster_smem();
  return true;
}

// Ring of claimed items of this CTA's cluster in the work queue `wq`: ring
// FIRST + blockIdx.x / CTAS (CTAS: CTAs per cluster).
template <int CTAS, int FIRST>
__device__ __forceinline__ unsigned long long* queue_ring(unsigned long long* wq) {
  return wq + 32 + static_cast<size_t>(FIRST + blockIdx.x / CTAS) * kQueueRing;
}

// Work item k of a persistent cluster's walk, read from the cluster's ring
// (entry k mod kQueueRing holds (k + 1) << 32 | pair index, written by the
// cluster's claimer with a release store): the pair index, or -1 past the
// walk's end (an index >= npairs) or when the bounded wait gives up (the same
// give-up rules as wait_bar).  Called once per item and role, so kept out of
// line (the roles' tile loops need their registers).
template <int CTAS, int FIRST>
__device__ __noinline__ int claimed(const Ctx c, unsigned long long* wq, int k, int npairs) {
  const unsigned long long* e = queue_ring<CTAS, FIRST>(wq) + (k & (kQueueRing - 1));
  const unsigned long long tag = static_cast<unsigned long long>(k + 1);
  uint32_t it = 0;
  uint64_t t0 = 0;
  while (true) {
    const unsigned long long v = tc::ld_acquire_gpu_u64(e);
    if ((v >> 32) == tag) {
      const uint32_t idx = static_cast<uint32_t>(v);
      return idx < static_cast<uint32_t>(npairs) ? static_cast<int>(idx) : -1;
    }
    if ((++it & 63u) == 0) {
      if (*c.abort || *reinterpret_cast<volatile int32_t*>(c.status)) {
        *c.abort = 1;
        return -1;
      }
      const uint64_t now = tc::global_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > WAIT_NS) {
        *c.abort = 1;
        atomicCAS(c.status, 0, static_cast<int32_t>(RK_ERR_DEVICE_TIMEOUT));
        return -1;
      }
    }
  }
}

// Bounded wait that ignores the abort flag (drains work in flight).
__device__ __forceinline__ void drain_bar(const Ctx& c, int i, uint32_t parity,
                                          uint64_t limit_ns = WAIT_NS) {
  uint64_t* b = c.bar + i;
  const uint64_t t0 = tc::global_ns();
  while (!tc::mbar_try_wait(b, parity)) {
    if (tc::global_ns() - t0 > limit_ns) {
      atomicCAS(c.status, 0, static_cast<int32_t>(RK_ERR_DEVICE_TIMEOUT));
      return;
    }
  }
}

struct RowInfo {
  int p;       // absolute row, -1 if the lane is unused
  int head;
  bool glob;   // Global visibility rule (k <= p), else Local (sink u [p - w, p])
  bool store;  // written by the epilogue
  int64_t frow;
};

// The query pair of TMEM lane m of tile t.  kind 0: row t.p0 + m % R of
// Global head m / R (R = 128 / HG).  kind 1: row t.p0 (m < H) or t.p1 of
// head m % H, stored only for Local heads.  Bit 0 of t.pad marks a tile
// without work (every lane unused).
__device__ __forceinline__ RowInfo row_info(const KernelArgs& a, const TcTile& t,
                                            const DevReq& rq, int m) {
  RowInfo r;
  const bool idle = (t.pad & 1) != 0;
  if (t.kind == 0) {
    const int R = a.rows_per_gtile;
    const int hi = m / R, ri = m - hi * R;
    const bool v = !idle && ri < t.p1 && hi < a.num_global;
    r.p = v ? t.p0 + ri : -1;
    r.head = v ? a.global_heads[hi] : 0;
    r.glob = true;
    r.store = v;
  } else {
    const int ri = m / a.H, h = m - ri * a.H;
    const int pr = idle ? -1 : ((ri == 0) ? t.p0 : t.p1);
    r.p = pr;
    r.head = h;
    r.glob = false;
    r.store = pr >= 0 && a.head_role[h] == 0;
  }
  r.frow = r.p >= 0 ? rq.row_base + (r.p - rq.q_row_begin) : -1;
  return r;
}

// Bit i set for each offset base + i (i < 32) inside [lo, hi).
__device__ __forceinline__ uint32_t span_bits(int lo, int hi, int base) {
  const int l = min(max(lo - base, 0), 32), h = min(max(hi - base, 0), 32);
  const uint32_t mh = h >= 32 ? 0xffffffffu : ((1u << h) - 1u);
  const uint32_t ml = l >= 32 ? 0xffffffffu : ((1u << l) - 1u);
  return mh & ~ml;
}

// Online softmax of one 128-key tile for one query pair, with its scores
// s[q4][i] (key k0 + 32 q4 + i, fp32 bits) from tensor memory (RedKnot-MLA
// paper, RoPE-orthogonality paragraph: the running max, sum and output carry
// across the key walk).  Keys the pair does not see become -inf (Global: k <=
// p; Local: sink u [p - w, p], RedKnot blog "Insight 1").  The running max
// (log2 domain) is raised only when the tile's max exceeds it by more than
// 2^8; the returned factor alpha (1 otherwise) rescales the earlier sum and
// output.  P = 2^(s * scale * log2 e - max) is left as bf16 pairs in s[0] and
// s[1] (keys 2w, 2w + 1 in word w = 16 q4 + i of s[q4 >> 1]).  The 4-CTA
// kernel and the side kernel beside it both use this, so a pair's P, sum and
// output are the same whichever of them takes it.
__device__ __forceinline__ float softmax_tile(uint32_t (&s)[4][32], const KeyTile& kt,
                                              const RowInfo& ri, int sink, int window,
                                              float sl2, float& m_run, float& l_run) {
  constexpr int TNK = 128;
  const int p = ri.p;
  const bool full = kt.k1 - kt.k0 == TNK && kt.k0 + TNK - 1 <= p &&
                    (ri.glob || kt.k0 >= p - window || kt.k0 + TNK <= sink);
  float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  if (__all_sync(0xffffffffu, full)) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
      for (int i = 0; i < 32; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(s[q4][i]));
  } else {
    // visible keys as offsets from k0: [0, a_hi) u [b_lo, hi) (a Global
    // head: [0, hi)), one bit per key of each 32-key group
    const int hi = min(max(min(kt.k1, p + 1) - kt.k0, 0), TNK);
    const int a_hi = ri.glob ? hi : min(hi, max(sink - kt.k0, 0));
    const int b_lo = ri.glob ? hi : max(p - window - kt.k0, 0);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const uint32_t msk = span_bits(0, a_hi, 32 * q4) | span_bits(b_lo, hi, 32 * q4);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float x = ((msk >> i) & 1u) ? __uint_as_float(s[q4][i]) : -INFINITY;
        s[q4][i] = __float_as_uint(x);
        mx4[i & 3] = fmaxf(mx4[i & 3], x);
      }
    }
  }
  const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
  float alpha = 1.f;
  if (mx > m_run + 8.f) {  // lazy rescale: only when the max grows by more than 2^8
    if (m_run != -INFINITY) alpha = fast_exp2(m_run - mx);
    m_run = mx;
  }
  const float nb = (m_run == -INFINITY) ? 0.f : -m_run;
  float ls4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float p0 = fast_exp2(fmaf(__uint_as_float(s[q4][2 * i]), sl2, nb));
      const float p1 = fast_exp2(fmaf(__uint_as_float(s[q4][2 * i + 1]), sl2, nb));
      ls4[i & 3] += p0 + p1;
      s[q4 >> 1][16 * (q4 & 1) + i] = pack_bf16x2(p0, p1);
    }
  }
  // explicit fused multiply-adds here and in lse_of: the kernels that share
  // this arithmetic get the same roundings whatever the compiler contracts
  l_run = fmaf(l_run, alpha, (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
  return alpha;
}

// Natural-log LSE of a query pair from its running max (log2 domain) and sum.
__device__ __forceinline__ float lse_of(float m_run, float l_run) {
  return fmaf(m_run, 0.6931471805599453f, logf(l_run));
}

// Turn the 16 rope pairs held in o[0..31] (32 consecutive output columns:
// pairs h0 .. h0 + 15 of the rope slice) by R(delta_a - delta_b), from the
// cos / sin tables of the two frames (float4 k: pairs 2k and 2k + 1).  The
// angles are formed here, for these 16 pairs only, to keep them out of the
// registers of the loops around.  Shared by the 4-CTA kernel and the side
// kernel beside it, so that both turn a pair's output the same way.
__device__ __forceinline__ void turn16(uint32_t (&o)[32], const float4* ca, const float4* cb, int h0) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const float4 x = __ldg(ca + h0 / 2 + u), y = __ldg(cb + h0 / 2 + u);
    const float c0 = fmaf(x.x, y.x, x.y * y.y), s0 = fmaf(x.y, y.x, -x.x * y.y);
    const float c1 = fmaf(x.z, y.z, x.w * y.w), s1 = fmaf(x.w, y.z, -x.z * y.w);
    const float a0 = __uint_as_float(o[4 * u]), b0 = __uint_as_float(o[4 * u + 1]);
    const float a1 = __uint_as_float(o[4 * u + 2]), b1 = __uint_as_float(o[4 * u + 3]);
    o[4 * u] = __float_as_uint(a0 * c0 - b0 * s0);
    o[4 * u + 1] = __float_as_uint(fmaf(a0, s0, b0 * c0));
    o[4 * u + 2] = __float_as_uint(a1 * c1 - b1 * s1);
    o[4 * u + 3] = __float_as_uint(fmaf(a1, s1, b1 * c1));
  }
}
// Turn the same 16 pairs by R(delta_frame - p): the frame's cos / sin table
// `ca` and the row position p's cos / sin of p theta from the two-level table
// (ph: the 256-multiple part, pl: the remainder), for the epilogue.
__device__ __forceinline__ void restore16(uint32_t (&o)[32], const float4* ca, const float4* ph,
                                          const float4* pl, int h0) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const float4 x = __ldg(ca + h0 / 2 + u), h = __ldg(ph + h0 / 2 + u), l = __ldg(pl + h0 / 2 + u);
    // cos / sin of p theta for pairs h0 + 2u, + 1
    const float pc0 = fmaf(h.x, l.x, -h.y * l.y), ps0 = fmaf(h.y, l.x, h.x * l.y);
    const float pc1 = fmaf(h.z, l.z, -h.w * l.w), ps1 = fmaf(h.w, l.z, h.z * l.w);
    const float c0 = fmaf(x.x, pc0, x.y * ps0), s0 = fmaf(x.y, pc0, -x.x * ps0);
    const float c1 = fmaf(x.z, pc1, x.w * ps1), s1 = fmaf(x.w, pc1, -x.z * ps1);
    const float a0 = __uint_as_float(o[4 * u]), b0 = __uint_as_float(o[4 * u + 1]);
    const float a1 = __uint_as_float(o[4 * u + 2]), b1 = __uint_as_float(o[4 * u + 3]);
    o[4 * u] = __float_as_uint(a0 * c0 - b0 * s0);
    o[4 * u + 1] = __float_as_uint(fmaf(a0, s0, b0 * c0));
    o[4 * u + 2] = __float_as_uint(a1 * c1 - b1 * s1);
    o[4 * u + 3] = __float_as_uint(fmaf(a1, s1, b1 * c1));
  }
}

// q_rope' = R(-delta) q_rope of one row (RedKnot-MLA paper, RoPE-orthogonality
// paragraph: the query turns by -delta_i instead of rewriting the cache) as
// bf16 hi and lo parts, written to this thread's TMEM lane at columns rh..
// and rl.. (rotation pair j in column j).  The row's q_rope (`src`, 64 bf16)
// is re-read from global memory each time; an unused lane (src == nullptr)
// writes zeros.
__device__ __forceinline__ void write_rope(uint32_t lane_taddr, uint32_t rh, uint32_t rl,
                                           const uint16_t* src, const float* cs) {
  uint32_t raw[32];
  if (src) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint4 v = __ldg(s4 + u);
      raw[4 * u] = v.x;
      raw[4 * u + 1] = v.y;
      raw[4 * u + 2] = v.z;
      raw[4 * u + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < 32; ++u) raw[u] = 0;
  }
  uint32_t hi[32];
#pragma unroll
  for (int jj = 0; jj < 32; ++jj) {
    const float x = __uint_as_float(raw[jj] << 16), y = __uint_as_float(raw[jj] & 0xffff0000u);
    const float co = __ldg(cs + 2 * jj), si = __ldg(cs + 2 * jj + 1);
    const float xr = fmaf(x, co, y * si), yr = fmaf(-x, si, y * co);
    hi[jj] = pack_bf16x2(xr, yr);
    raw[jj] = pack_bf16x2(xr - __uint_as_float(hi[jj] << 16),
                          yr - __uint_as_float(hi[jj] & 0xffff0000u));
  }
  tc::tmem_st32(lane_taddr + rh, hi);
  tc::tmem_st32(lane_taddr + rl, raw);
  tc::tmem_wait_st();
}

// TMA views of q (bf16 [rows, H, d_k], d_k = 64 (NCH + 1): NCH nope chunks
// then the rope chunk) for loading a tile's nope part chunk-major into shared
// memory (NCH chunks of 128 lanes x 64 dims, 128-byte swizzled).
struct QMaps {
  CUtensorMap g5;   // Global, one Global head per group: (64, rows, groups, NCH chunks, in-group)
  CUtensorMap g3;   // Global, any roles: (d_k, H, rows), box (64, 1, R)
  CUtensorMap l4;   // Local, H = 128: (64, H, NCH chunks, rows), box (64, 128, NCH, 1)
  CUtensorMap l3;   // Local, any H: (d_k, H, rows), box (64, H, 1)
};

inline cudaError_t make_qmaps(const rk_seg_attn_plan_s& p, const KernelArgs& a, const void* q,
                              QMaps& qm) {
  qm = QMaps{};
  const uint64_t H = static_cast<uint64_t>(p.H), rows = static_cast<uint64_t>(p.info.rows);
  const uint64_t dk = static_cast<uint64_t>(p.d_nope + p.d_rope), rb = 2 * dk;  // row bytes
  const uint32_t nch = static_cast<uint32_t>(p.d_nope / 64);
  const uint32_t R = static_cast<uint32_t>(a.rows_per_gtile > 0 ? a.rows_per_gtile : 8);
  if (a.g_ingroup >= 0) {  // the whole Global tile in one box
    const uint64_t G = H / 8;
    const uint64_t dims[5] = {64, rows, G, nch, 8};
    const uint64_t strides[4] = {H * rb, 8 * rb, 128, rb};
    const uint32_t box[5] = {64, R, static_cast<uint32_t>(G), nch, 1};
    if (!make_tmap_bf16(&qm.g5, q, 5, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {dk, H, rows};
    const uint64_t strides[2] = {rb, H * rb};
    const uint32_t boxg[3] = {64, 1, R};
    const uint32_t boxl[3] = {64, static_cast<uint32_t>(H), 1};
    if (!make_tmap_bf16(&qm.g3, q, 3, dims, strides, boxg)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&qm.l3, q, 3, dims, strides, boxl)) return cudaErrorInvalidValue;
  }
  if (H == 128) {
    const uint64_t dims[4] = {64, H, nch, rows};
    const uint64_t strides[3] = {rb, 128, H * rb};
    const uint32_t box[4] = {64, static_cast<uint32_t>(H), nch, 1};
    if (!make_tmap_bf16(&qm.l4, q, 4, dims, strides, box)) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

// Issue the TMA loads of tile t's queries (NCH x 16 KB) into `qdst`, from
// maps that make_qmaps built for a plan with d_nope = 64 NCH.  PAIR: the
// copies complete on the barrier at cluster address `bar` (cta_group::2
// form, the barrier may be the peer's); otherwise on this CTA's barrier at
// shared address `bar`.
template <bool PAIR, int NCH = 8>
__device__ __forceinline__ void load_q_tile(const KernelArgs& a, const QMaps& qm, const TcTile& t,
                                            const DevReq& rq, uint32_t qdst, uint32_t bar) {
  auto ld3 = [&](uint32_t dst, const CUtensorMap* m, int32_t x, int32_t y, int32_t z) {
    if (PAIR)
      tc::tma_load_3d_2sm(dst, m, bar, x, y, z);
    else
      tc::tma_load_3d_u32(dst, m, bar, x, y, z);
  };
  if (t.kind == 0) {
    const int32_t fr = static_cast<int32_t>(rq.row_base + (t.p0 - rq.q_row_begin));
    if (a.g_ingroup >= 0) {
      if (PAIR)
        tc::tma_load_5d_2sm(qdst, &qm.g5, bar, 0, fr, 0, 0, a.g_ingroup);
      else
        tc::tma_load_5d_u32(qdst, &qm.g5, bar, 0, fr, 0, 0, a.g_ingroup);
    } else {
      const int R = a.rows_per_gtile;
      for (int ch = 0; ch < NCH; ++ch)
        for (int hi = 0; hi < a.num_global; ++hi)
          ld3(qdst + ch * 16384 + hi * R * 128, &qm.g3, 64 * ch, a.global_heads[hi], fr);
    }
  } else if (a.H == 128) {
    const int32_t fr = static_cast<int32_t>(rq.row_base + (t.p0 - rq.q_row_begin));
    if (PAIR)
      tc::tma_load_4d_2sm(qdst, &qm.l4, bar, 0, 0, 0, fr);
    else
      tc::tma_load_4d_u32(qdst, &qm.l4, bar, 0, 0, 0, fr);
  } else {
    const int rows_per = 128 / a.H;
    for (int ch = 0; ch < NCH; ++ch)
      for (int ri = 0; ri < rows_per; ++ri) {
        const int pr = (ri == 0 || t.p1 < 0) ? t.p0 : t.p1;
        const int32_t fr = static_cast<int32_t>(rq.row_base + (pr - rq.q_row_begin));
        ld3(qdst + ch * 16384 + ri * a.H * 128, &qm.l3, 64 * ch, 0, fr);
      }
  }
}

}  // namespace tt
}  // namespace rk
