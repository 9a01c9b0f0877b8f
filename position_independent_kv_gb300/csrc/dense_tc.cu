// Prefill-style tiles on the sm_100-family tensor path (tcgen05 + TMEM + TMA).
//
// One tile = 128 query pairs (Global: 128/HG consecutive rows x the HG
// Global heads; Local: one or two protected rows x every head, only the
// Local heads stored) over the tile's key range.  Two CTAs run each tile,
// one per half of d_v (256 output columns each), because the fp32 output of
// 128 pairs x 512 columns alone would fill tensor memory.
//
// Per CTA (256 threads, warp-specialised):
//   warp 0  TMA producer: the 8 nope chunks of Q once (128 rows x 64 dims,
//           128-byte swizzle), then the latent stream through a 4-slot ring
//           of 16 KB chunks (128 keys x 64 dims): for key tile j the 9 chunks
//           of the score contraction, then (one tile later) the 4 chunks of
//           this CTA's d_v half again for P.V.
//   warp 1  MMA issuer: S_j = Q K^T (M=128, N=128, K = 512 + 64 hi + 64 lo)
//           into one of two TMEM score buffers, P.V (A = P from TMEM, B =
//           the V chunk in MN-major form) into the 256 fp32 output columns.
//   warps 2-3  query rotation: per segment, q_rope' = R(-delta) q_rope (fp32
//           from the fp64-derived table) written as bf16 hi + lo chunks
//           (RedKnot-MLA paper, RoPE-orthogonality paragraph).
//   warps 4-7  online softmax, one thread per query pair (TMEM lane): masks
//           (Global k <= p; Local sink u [p - w, p], RedKnot blog "Insight
//           1"), running max in the log2 domain with a lazy rescale of the
//           output when the max grows by more than 2^8, P (bf16) written
//           over the score buffer, and the epilogue (normalise, bf16 store,
//           LSE).  The running state carries across segments: each segment
//           boundary is a log-sum-exp merge point.
// Every wait is bounded in time; on expiry the CTA records
// RK_ERR_DEVICE_TIMEOUT, every role stops, the producer waits (bounded) for
// its copies in flight and TMEM is released only after the MMA pipe drains.

#include "tc_ptx.cuh"
#include "tmap.h"

namespace rk {
namespace {

constexpr int TM = 128;
constexpr int TNK = 128;
constexpr uint32_t CHUNK = 16384;
constexpr int RING = 4;
constexpr int THREADS = 256;
constexpr uint64_t WAIT_NS = 2000000000ull;

constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_HI = 8 * CHUNK;
constexpr uint32_t OFF_LO = 9 * CHUNK;
constexpr uint32_t OFF_RING = 10 * CHUNK;
constexpr uint32_t OFF_BAR = OFF_RING + RING * CHUNK;
enum {
  B_FULL = 0,
  B_EMPTY = RING,
  B_QFULL = 2 * RING,
  B_SFULL = 2 * RING + 1,   // 2
  B_PREADY = 2 * RING + 3,  // 2
  B_ODONE = 2 * RING + 5,
  B_RREADY,
  B_RFREE,
  B_FINAL,
  NBAR
};
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;

constexpr uint32_t T_O = 0, T_S0 = 256, T_S1 = 384;

struct Ctx {
  uint64_t* bar;
  volatile uint32_t* abort;
  int32_t* status;
};

// Bounded wait; also gives up as soon as another role of this CTA, or any
// CTA of the launch, has recorded an error.
__device__ __forceinline__ bool wait_bar(const Ctx& c, int i, uint32_t parity) {
  uint64_t* b = c.bar + i;
  uint32_t it = 0;
  uint64_t t0 = 0;
  while (!tc::mbar_try_wait(b, parity)) {
    if ((++it & 63u) == 0) {
      if (*c.abort || *reinterpret_cast<volatile int32_t*>(c.status)) {
        *c.abort = 1;
        return false;
      }
      const uint64_t now = tc::global_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > WAIT_NS) {
        *c.abort = 1;
        atomicCAS(c.status, 0, static_cast<int32_t>(RK_ERR_DEVICE_TIMEOUT));
        return false;
      }
    }
  }
  return true;
}

// Bounded wait that ignores the abort flag (used to drain copies in flight).
__device__ __forceinline__ void drain_bar(const Ctx& c, int i, uint32_t parity) {
  uint64_t* b = c.bar + i;
  const uint64_t t0 = tc::global_ns();
  while (!tc::mbar_try_wait(b, parity)) {
    if (tc::global_ns() - t0 > WAIT_NS) {
      atomicCAS(c.status, 0, static_cast<int32_t>(RK_ERR_DEVICE_TIMEOUT));
      return;
    }
  }
}

struct RowInfo {
  int p;       // absolute row, -1 if the pair is unused
  int head;
  bool glob;   // Global visibility rule
  bool store;  // written by the epilogue
  int64_t frow;
};

__device__ __forceinline__ RowInfo row_info(const KernelArgs& a, const TcTile& t,
                                            const DevReq& rq, int m) {
  RowInfo r;
  if (t.kind == 0) {
    const int R = a.rows_per_gtile;
    const int hi = m / R, ri = m - hi * R;
    const bool v = ri < t.p1 && hi < a.num_global;
    r.p = v ? t.p0 + ri : -1;
    r.head = v ? a.global_heads[hi] : 0;
    r.glob = true;
    r.store = v;
  } else {
    const int ri = m / a.H, h = m - ri * a.H;
    const int pr = (ri == 0) ? t.p0 : t.p1;
    r.p = pr;
    r.head = h;
    r.glob = false;
    r.store = pr >= 0 && a.head_role[h] == 0;
  }
  r.frow = r.p >= 0 ? rq.row_base + (r.p - rq.q_row_begin) : -1;
  return r;
}

__global__ void __launch_bounds__(THREADS, 1)
    dense_tc_kernel(const KernelArgs a, const __grid_constant__ CUtensorMap tmQg,
                    const __grid_constant__ CUtensorMap tmQl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  const Ctx c{bar, reinterpret_cast<volatile uint32_t*>(misc + 1), a.status};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int half = blockIdx.x & 1;
  const TcTile t = a.tc_tiles[blockIdx.x >> 1];
  const DevReq rq = a.reqs[t.req];
  const DevSeg* segs = a.segs + rq.seg_first;
  const int nseg = rq.seg_count;
  const int r0hi = t.sink_hi, r1lo = t.win_lo, r1hi = t.key_hi;

  if (tid == 0) {
    for (int i = 0; i < RING; ++i) {
      tc::mbar_init(&bar[B_FULL + i], 1);
      tc::mbar_init(&bar[B_EMPTY + i], 1);
    }
    tc::mbar_init(&bar[B_QFULL], 1);
    tc::mbar_init(&bar[B_SFULL], 1);
    tc::mbar_init(&bar[B_SFULL + 1], 1);
    tc::mbar_init(&bar[B_PREADY], 128);
    tc::mbar_init(&bar[B_PREADY + 1], 128);
    tc::mbar_init(&bar[B_ODONE], 1);
    tc::mbar_init(&bar[B_RREADY], 2);
    tc::mbar_init(&bar[B_RFREE], 1);
    tc::mbar_init(&bar[B_FINAL], 1);
    misc[1] = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(misc, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = misc[0];

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      tc::prefetch_tmap(&tmQg);
      tc::prefetch_tmap(&tmQl);
      tc::mbar_arrive_expect_tx(&bar[B_QFULL], 8 * CHUNK);
      for (int ch = 0; ch < 8; ++ch) {
        const uint32_t dst = smem_u32(sm + OFF_Q + ch * CHUNK);
        if (t.kind == 0) {
          const int R = a.rows_per_gtile;
          const int64_t fr = rq.row_base + (t.p0 - rq.q_row_begin);
          for (int hi = 0; hi < a.num_global; ++hi)
            tc::tma_load_3d(dst + hi * R * 128, &tmQg, &bar[B_QFULL], 64 * ch,
                            a.global_heads[hi], static_cast<int32_t>(fr));
        } else {
          const int rows_per = TM / a.H;
          for (int ri = 0; ri < rows_per; ++ri) {
            const int pr = (ri == 0 || t.p1 < 0) ? t.p0 : t.p1;
            const int64_t fr = rq.row_base + (pr - rq.q_row_begin);
            tc::tma_load_3d(dst + ri * a.H * 128, &tmQl, &bar[B_QFULL], 64 * ch, 0,
                            static_cast<int32_t>(fr));
          }
        }
      }
      uint32_t cnt = 0;
      bool ok = true;
      auto load = [&](const KeyTile& kt, int ch) {
        const int slot = cnt % RING;
        const uint32_t ph = (cnt / RING) & 1;
        if (!wait_bar(c, B_EMPTY + slot, ph ^ 1)) return false;
        tc::mbar_arrive_expect_tx(&bar[B_FULL + slot], CHUNK);
        tc::tma_load_2d(smem_u32(sm + OFF_RING + slot * CHUNK), a.segmaps + rq.seg_first + kt.j,
                        &bar[B_FULL + slot], 64 * ch, kt.k0 - segs[kt.j].delta);
        ++cnt;
        return true;
      };
      KeyTile cur{0, 0, 0, -1}, prev{0, 0, 0, -1};
      bool have = next_key_tile<TNK>(cur, segs, nseg, 0, r0hi, r1lo, r1hi);
      bool has_prev = false;
      while (ok && (have || has_prev)) {
        if (have)
          for (int ch = 0; ch < 9 && ok; ++ch) ok = load(cur, ch);
        if (has_prev && ok)
          for (int v = 0; v < 4 && ok; ++v) ok = load(prev, 4 * half + v);
        prev = cur;
        has_prev = have;
        if (have) have = next_key_tile<TNK>(cur, segs, nseg, 0, r0hi, r1lo, r1hi);
      }
      // copies in flight must land before the CTA may exit
      drain_bar(c, B_QFULL, 0);
      for (uint32_t k = (cnt > RING ? cnt - RING : 0); k < cnt; ++k)
        drain_bar(c, B_FULL + k % RING, (k / RING) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      bool ok = wait_bar(c, B_QFULL, 0);
      tc::tc_fence_after();
      const uint32_t idS = tc::idesc_bf16(128, 128, false, false);
      const uint32_t idPV = tc::idesc_bf16(128, 64, false, true);
      const uint32_t qa = smem_u32(sm + OFF_Q), ha = smem_u32(sm + OFF_HI),
                     la = smem_u32(sm + OFF_LO), ra = smem_u32(sm + OFF_RING);
      uint32_t cnt = 0;
      int j = 0, jprev = -1, cur_seg = -1, sidx = -1;
      KeyTile cur{0, 0, 0, -1};
      bool have = next_key_tile<TNK>(cur, segs, nseg, 0, r0hi, r1lo, r1hi);
      bool has_prev = false;
      while (ok && (have || has_prev)) {
        if (have) {
          const uint32_t Sb = tbase + ((j & 1) ? T_S1 : T_S0);
          if (cur.j != cur_seg) {
            ++sidx;
            ok = wait_bar(c, B_RREADY, sidx & 1);
            tc::tc_fence_after();
            cur_seg = cur.j;
          }
          for (int ch = 0; ch < 9 && ok; ++ch) {
            const int slot = cnt % RING;
            ok = wait_bar(c, B_FULL + slot, (cnt / RING) & 1);
            if (!ok) break;
            tc::tc_fence_after();
            const uint32_t kb = ra + slot * CHUNK;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t bd = tc::sdesc_sw128(kb + 32 * k, 16, 1024);
              if (ch < 8) {
                tc::mma_ss(Sb, tc::sdesc_sw128(qa + ch * CHUNK + 32 * k, 16, 1024), bd, idS,
                           (ch | k) != 0);
              } else {
                tc::mma_ss(Sb, tc::sdesc_sw128(ha + 32 * k, 16, 1024), bd, idS, 1);
                tc::mma_ss(Sb, tc::sdesc_sw128(la + 32 * k, 16, 1024), bd, idS, 1);
              }
            }
            tc::mma_commit(&bar[B_EMPTY + slot]);
            ++cnt;
          }
          if (!ok) break;
          tc::mma_commit(&bar[B_SFULL + (j & 1)]);
          KeyTile nx = cur;
          const bool hn = next_key_tile<TNK>(nx, segs, nseg, 0, r0hi, r1lo, r1hi);
          if (!hn || nx.j != cur.j) tc::mma_commit(&bar[B_RFREE]);
        }
        if (has_prev) {
          const int pb = jprev & 1;
          const uint32_t Pb = tbase + (pb ? T_S1 : T_S0);
          ok = wait_bar(c, B_PREADY + pb, (jprev >> 1) & 1);
          if (!ok) break;
          tc::tc_fence_after();
          for (int v = 0; v < 4 && ok; ++v) {
            const int slot = cnt % RING;
            ok = wait_bar(c, B_FULL + slot, (cnt / RING) & 1);
            if (!ok) break;
            tc::tc_fence_after();
            const uint32_t vb = ra + slot * CHUNK;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              tc::mma_ts(tbase + T_O + 64 * v, Pb + 8 * k, tc::sdesc_sw128(vb + 2048 * k, 1024, 1024),
                         idPV, (jprev > 0 || k > 0) ? 1u : 0u);
            tc::mma_commit(&bar[B_EMPTY + slot]);
            ++cnt;
          }
          if (!ok) break;
          tc::mma_commit(&bar[B_ODONE]);
        }
        has_prev = have;
        jprev = j;
        if (have) {
          have = next_key_tile<TNK>(cur, segs, nseg, 0, r0hi, r1lo, r1hi);
          ++j;
        }
      }
      tc::mma_commit(&bar[B_FINAL]);
    }
  } else if (warp == 2 || warp == 3) {
    // -------------------------------------------------- query rotation ----
    // warp 2 rotates rows 0..63, warp 3 rows 64..127
    const int mbase = (warp - 2) * 64;
    uint32_t raw[2][32];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const RowInfo ri = row_info(a, t, rq, mbase + lane + 32 * i);
      if (ri.p >= 0) {
        const uint4* src = reinterpret_cast<const uint4*>(a.q + (ri.frow * a.H + ri.head) * 576 + 512);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = src[u];
          raw[i][4 * u] = v.x;
          raw[i][4 * u + 1] = v.y;
          raw[i][4 * u + 2] = v.z;
          raw[i][4 * u + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int u = 0; u < 32; ++u) raw[i][u] = 0;
      }
    }
    int cur_seg = -1, sidx = -1;
    bool ok = true;
    KeyTile kt{0, 0, 0, -1};
    while (ok && next_key_tile<TNK>(kt, segs, nseg, 0, r0hi, r1lo, r1hi)) {
      if (kt.j == cur_seg) continue;
      ++sidx;
      if (sidx > 0) ok = __all_sync(0xffffffffu, wait_bar(c, B_RFREE, (sidx - 1) & 1));
      if (!ok) break;
      const float* cs = a.rope_cs + static_cast<int64_t>(rq.seg_first + kt.j) * 64;
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const float co = __ldg(cs + 2 * jj), si = __ldg(cs + 2 * jj + 1);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint32_t m = mbase + lane + 32 * i;
          const float x = __uint_as_float(raw[i][jj] << 16);
          const float y = __uint_as_float(raw[i][jj] & 0xffff0000u);
          const float xr = fmaf(x, co, y * si);
          const float yr = fmaf(-x, si, y * co);
          const uint32_t h2 = pack_bf16x2(xr, yr);
          const float xh = __uint_as_float(h2 << 16), yh = __uint_as_float(h2 & 0xffff0000u);
          const uint32_t off = tc::sw128_offset(m, 2 * jj);
          *reinterpret_cast<uint32_t*>(sm + OFF_HI + off) = h2;
          *reinterpret_cast<uint32_t*>(sm + OFF_LO + off) = pack_bf16x2(xr - xh, yr - yh);
        }
      }
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[B_RREADY]);
      cur_seg = kt.j;
    }
  } else if (warp >= 4) {
    // --------------------------------------------------- online softmax ---
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const RowInfo ri = row_info(a, t, rq, m);
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = a.scale_log2;
    const int sink = a.sink, window = a.window;
    float m_run = -INFINITY, l_run = 0.f;
    int j = 0;
    bool ok = true;
    KeyTile kt{0, 0, 0, -1};
    while (ok && next_key_tile<TNK>(kt, segs, nseg, 0, r0hi, r1lo, r1hi)) {
      const int b = j & 1;
      const uint32_t Sb = tbase + lane_off + (b ? T_S1 : T_S0);
      ok = __all_sync(0xffffffffu, wait_bar(c, B_SFULL + b, (j >> 1) & 1));
      if (!ok) break;
      tc::tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tc::tmem_ld32(Sb + 32 * q4, s[q4]);
      tc::tmem_wait_ld();
      float mx = -INFINITY;
      const int p = ri.p;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int key = kt.k0 + 32 * q4 + i;
          bool vis = key < kt.k1 && key <= p;
          if (!ri.glob) vis = vis && (key < sink || key >= p - window);
          const float x = vis ? __uint_as_float(s[q4][i]) * sl2 : -INFINITY;
          s[q4][i] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      }
      bool need = false;
      float alpha = 1.f;
      if (mx > m_run + 8.f) {
        if (m_run != -INFINITY) {
          need = true;
          alpha = fast_exp2(m_run - mx);
        }
        m_run = mx;
      }
      const float base = (m_run == -INFINITY) ? 0.f : m_run;
      float ls = 0.f;
      // P in place: pair i of column block q4 goes to word 16 * q4 + i, i.e.
      // s[q4 >> 1][16 * (q4 & 1) + i]; every word is read before it is written
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = fast_exp2(__uint_as_float(s[q4][2 * i]) - base);
          const float p1 = fast_exp2(__uint_as_float(s[q4][2 * i + 1]) - base);
          ls += p0 + p1;
          s[q4 >> 1][16 * (q4 & 1) + i] = pack_bf16x2(p0, p1);
        }
      }
      l_run = l_run * alpha + ls;
      tc::tmem_st32(Sb, s[0]);
      tc::tmem_st32(Sb + 32, s[1]);
      tc::tmem_wait_st();
      if (__any_sync(0xffffffffu, need)) {
        if (j >= 1) ok = __all_sync(0xffffffffu, wait_bar(c, B_ODONE, (j - 1) & 1));
        if (ok) {
          tc::tc_fence_after();
          const uint32_t Ob = tbase + lane_off + T_O;
#pragma unroll 1
          for (int q8 = 0; q8 < 8; ++q8) {
            uint32_t o[32];
            tc::tmem_ld32(Ob + 32 * q8, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tc::tmem_st32(Ob + 32 * q8, o);
          }
          tc::tmem_wait_st();
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&bar[B_PREADY + b]);
      ++j;
    }
    // ---- epilogue ----
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(c, B_FINAL, 0));
    tc::tc_fence_after();
    if (ok) {
      const bool st = ri.store && l_run > 0.f;
      const float inv = st ? 1.f / l_run : 0.f;
      uint16_t* dst = st ? a.out + (ri.frow * a.H + ri.head) * 512 + 256 * half : nullptr;
      const uint32_t Ob = tbase + lane_off + T_O;
#pragma unroll 1
      for (int q8 = 0; q8 < 8; ++q8) {
        uint32_t o[32];
        tc::tmem_ld32(Ob + 32 * q8, o);
        tc::tmem_wait_ld();
        if (st) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * q8);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * u + 0]) * inv, __uint_as_float(o[8 * u + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[8 * u + 2]) * inv, __uint_as_float(o[8 * u + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[8 * u + 4]) * inv, __uint_as_float(o[8 * u + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[8 * u + 6]) * inv, __uint_as_float(o[8 * u + 7]) * inv);
            d4[u] = v;
          }
        }
      }
      if (st && half == 0) a.lse[ri.frow * a.H + ri.head] = m_run * 0.6931471805599453f + logf(l_run);
    }
  }

  // ------------------------------------------------------------ teardown --
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    drain_bar(c, B_FINAL, 0);  // the MMA pipe is empty before TMEM is released
    tc::tc_fence_after();
    tc::tmem_dealloc(tbase, 512);
  }
}

}  // namespace

cudaError_t launch_dense_tc(const rk_seg_attn_plan_s& p, const KernelArgs& a, const void* q,
                            cudaStream_t s) {
  CUtensorMap tg{}, tl{};
  const uint64_t dims[3] = {576, static_cast<uint64_t>(p.H), static_cast<uint64_t>(p.info.rows)};
  const uint64_t strides[2] = {1152, static_cast<uint64_t>(p.H) * 1152};
  const uint32_t boxg[3] = {64, 1, static_cast<uint32_t>(a.rows_per_gtile > 0 ? a.rows_per_gtile : 8)};
  const uint32_t boxl[3] = {64, static_cast<uint32_t>(p.H), 1};
  if (!make_tmap_bf16(&tg, q, 3, dims, strides, boxg)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tl, q, 3, dims, strides, boxl)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(dense_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  const int64_t grid = 2 * static_cast<int64_t>(a.num_tc_tiles);
  dense_tc_kernel<<<static_cast<unsigned>(grid), THREADS, SMEM_BYTES, s>>>(a, tg, tl);
  return cudaGetLastError();
}

}  // namespace rk
