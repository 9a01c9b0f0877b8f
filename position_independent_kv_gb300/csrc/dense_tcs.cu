// Prefill-style tiles for small heads on the tensor path (tcgen05 + TMEM +
// TMA): d_nope = 128, d_rope = 32, V = c_nope (d_v = 128).
//
// One CTA per tile of 128 query pairs (the work list of the plan's generic
// tiles: kind 0 = rows x every Global head, row-major; kind 1 = a run of the
// flattened (protected row, Local head) list).  At this size every operand
// of a tile fits one SM, so there is no role split across CTAs:
//
//   tensor memory (512 columns): O (128, fp32) | S (128, fp32) | P (64, bf16
//   pairs) | Q nope (64, bf16 pairs) | q_rope' hi (16) | lo (16)
//
//   warp 0     TMA producer: each 128-key tile of the canonical latent
//              arrives as three 16 KB boxes of 64 dims x 128 keys (128-byte
//              swizzle) from a [n, 160] row-major map: dims 0-63, 64-127 and
//              128-159 (the last box's other 32 dims lie outside the map and
//              read as zero).  A slot stays resident until the P.V of its
//              tile: the two nope boxes are the value rows of the same keys.
//   warp 1     MMA issuer: S_j = Q K_j^T (A = Q nope, then q_rope' hi and
//              lo, all from tensor memory; B = the key boxes, K-major;
//              M = 128, N = 128), then O += P_{j-1} V_{j-1} (A = P from
//              tensor memory, B = the nope boxes read MN-major, N = 128).
//   warps 2-5  one thread per query pair (its TMEM lane): writes its query's
//              nope part into tensor memory, the rotated q_rope of each
//              segment the key walk enters (the query turns by -delta_i:
//              RedKnot-MLA paper, RoPE-orthogonality paragraph), loads S,
//              masks edge tiles (Global k <= p; Local sink u [p - w, p],
//              RedKnot blog "Insight 1"), keeps the running max in the log2
//              domain with a lazy rescale of O, writes P, and finally
//              normalises and stores O and the LSE.  The running state
//              carries across segments: each segment end is a log-sum-exp
//              merge point.
//
// Every wait is bounded in time; on expiry the CTA records
// RK_ERR_DEVICE_TIMEOUT, every role stops, the producer waits (bounded) for
// its copies in flight and tensor memory is released after the MMA pipe
// drains.

#include "tc_tile.cuh"

namespace rk {
namespace {

using tt::Ctx;
using tt::drain_bar;
using tt::wait_bar;

constexpr int TNK = 128;                 // keys per key tile
constexpr int DN = 128, DR = 32, DK = DN + DR, DV = DN;
constexpr uint32_t CHUNK = 16384;        // 128 keys x 64 bf16
constexpr int NBOX = 3;                  // dims 0-63, 64-127, 128-159 (+ zeros)
constexpr uint32_t SLOT = NBOX * CHUNK;
constexpr int RING = 3;
constexpr int THREADS = 192;

constexpr uint32_t OFF_RING = 0;
constexpr uint32_t OFF_BAR = OFF_RING + RING * SLOT;
enum { B_FULL = 0, B_EMPTY = RING, B_SFULL = 2 * RING, B_SFREE, B_PREADY, B_ODONE, B_FINAL, NBAR };
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");

constexpr uint32_t T_O = 0, T_S = 128, T_P = 256, T_Q = 320, T_RH = 384, T_RL = 400;

struct PairInfo {
  int p;        // absolute row, -1 if the lane is unused
  int head;
  bool glob;    // Global visibility rule (k <= p), else Local (sink u [p - w, p])
  int64_t frow; // flattened computed row
};

__device__ __forceinline__ PairInfo pair_info(const KernelArgs& a, const DenseTile& t,
                                              const DevReq& rq, int m) {
  PairInfo r{-1, 0, t.kind == 0, -1};
  if (t.kind == 0) {
    const int HG = a.num_global;
    const int ri = m / HG;
    if (ri < t.count) {
      r.p = t.first + ri;
      r.head = a.global_heads[m - ri * HG];
    }
  } else if (m < t.count) {
    const int i = t.first + m;
    const int lr = i / a.num_local;
    r.p = a.local_rows[lr];
    r.head = a.local_heads[i - lr * a.num_local];
  }
  if (r.p >= 0) r.frow = rq.row_base + (r.p - rq.q_row_begin);
  return r;
}

// q_rope' = R(-delta) q_rope of this lane's query (16 rotation pairs) as
// bf16 hi and lo parts: columns T_RH + j and T_RL + j hold pair j.  The 32
// columns are written in one store (hi then lo).  raw: the query's q_rope
// as 16 packed bf16 pairs (zeros for an unused lane); cs: the segment's
// (cos, sin) of delta * theta_j.
__device__ __forceinline__ void put_rope(uint32_t lane_taddr, const uint32_t (&raw)[16],
                                         const float* cs) {
  const float4* c4 = reinterpret_cast<const float4*>(cs);
  uint32_t w[32];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const float4 v = __ldg(c4 + u);  // pairs 2u, 2u + 1
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int jj = 2 * u + h;
      const float co = h ? v.z : v.x, si = h ? v.w : v.y;
      const float x = __uint_as_float(raw[jj] << 16);
      const float y = __uint_as_float(raw[jj] & 0xffff0000u);
      const float xr = fmaf(x, co, y * si), yr = fmaf(-x, si, y * co);
      const uint32_t hw = pack_bf16x2(xr, yr);
      w[jj] = hw;
      w[16 + jj] = pack_bf16x2(xr - __uint_as_float(hw << 16), yr - __uint_as_float(hw & 0xffff0000u));
    }
  }
  tc::tmem_st32(lane_taddr + T_RH, w);
}

__global__ void __launch_bounds__(THREADS, 1) dense_tcs_kernel(const KernelArgs a) {
  static_assert(T_RL == T_RH + 16, "hi and lo written as one 32-column store");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  const Ctx c{bar, reinterpret_cast<volatile uint32_t*>(misc + 1), a.status};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const DenseTile t = a.tiles[blockIdx.x];
  const DevReq rq = a.reqs[t.req];
  const DevSeg* segs = a.segs + rq.seg_first;
  const int nseg = rq.seg_count;
  const int r0hi = t.sink_hi, r1lo = t.win_lo, r1hi = t.key_hi;

  if (tid == 0) {
    for (int i = 0; i < RING; ++i) {
      tc::mbar_init(&bar[B_FULL + i], 1);
      tc::mbar_init(&bar[B_EMPTY + i], 1);
    }
    tc::mbar_init(&bar[B_SFULL], 1);
    tc::mbar_init(&bar[B_SFREE], 4);   // one arrival per lane warp
    tc::mbar_init(&bar[B_PREADY], 4);
    tc::mbar_init(&bar[B_ODONE], 1);
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
      uint32_t cnt = 0;
      bool ok = true;
      KeyTile cur{0, 0, 0, -1};
      bool have = next_key_tile<TNK>(cur, segs, nseg, 0, r0hi, r1lo, r1hi);
      while (ok && have) {
        const int slot = cnt % RING;
        ok = wait_bar(c, B_EMPTY + slot, ((cnt / RING) & 1) ^ 1);
        if (!ok) break;
        tc::mbar_arrive_expect_tx(&bar[B_FULL + slot], SLOT);
        const CUtensorMap* map = a.segmaps + kSegMaps * (rq.seg_first + cur.j);
        const int y = cur.k0 - segs[cur.j].delta;
#pragma unroll
        for (int b = 0; b < NBOX; ++b)
          tc::tma_load_2d(smem_u32(sm + OFF_RING + slot * SLOT + b * CHUNK), map,
                          &bar[B_FULL + slot], 64 * b, y);
        ++cnt;
        have = next_key_tile<TNK>(cur, segs, nseg, 0, r0hi, r1lo, r1hi);
      }
      // copies in flight must land before the CTA may exit
      for (uint32_t k = (cnt > RING ? cnt - RING : 0); k < cnt; ++k)
        drain_bar(c, B_FULL + k % RING, (k / RING) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      const uint32_t idS = tc::idesc_bf16(128, 128, false, false);
      const uint32_t idPV = tc::idesc_bf16(128, DV, false, true);
      const uint32_t ra = smem_u32(sm + OFF_RING);
      int j = 0, jprev = -1;
      bool ok = true;
      KeyTile cur{0, 0, 0, -1};
      bool have = next_key_tile<TNK>(cur, segs, nseg, 0, r0hi, r1lo, r1hi);
      bool has_prev = false;
      while (ok && (have || has_prev)) {
        if (have) {
          // the lanes have read S_{j-1} (and written Q and this segment's q_rope')
          ok = wait_bar(c, B_SFREE, j & 1);
          if (!ok) break;
          const int slot = j % RING;
          ok = wait_bar(c, B_FULL + slot, (j / RING) & 1);
          if (!ok) break;
          tc::tc_fence_after();
          const uint32_t base = ra + slot * SLOT;
#pragma unroll
          for (int cc = 0; cc < DN / 64; ++cc)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc::mma_ts(tbase + T_S, tbase + T_Q + 8 * (4 * cc + k),
                         tc::sdesc_sw128(base + cc * CHUNK + 32 * k, 16, 1024), idS,
                         (cc | k) != 0);
#pragma unroll
          for (int k = 0; k < DR / 16; ++k) {
            const uint64_t bd = tc::sdesc_sw128(base + (DN / 64) * CHUNK + 32 * k, 16, 1024);
            tc::mma_ts(tbase + T_S, tbase + T_RH + 8 * k, bd, idS, 1);
            tc::mma_ts(tbase + T_S, tbase + T_RL + 8 * k, bd, idS, 1);
          }
          tc::mma_commit(&bar[B_SFULL]);
        }
        if (has_prev) {
          ok = wait_bar(c, B_PREADY, jprev & 1);
          if (!ok) break;
          tc::tc_fence_after();
          const int slot = jprev % RING;
          const uint32_t base = ra + slot * SLOT;
          // B = V[16 keys x 128 dims]: the two nope boxes, 16 KB apart (LBO)
#pragma unroll
          for (int k = 0; k < TNK / 16; ++k)
            tc::mma_ts(tbase + T_O, tbase + T_P + 8 * k,
                       tc::sdesc_sw128(base + 2048 * k, CHUNK, 1024), idPV,
                       (jprev > 0 || k > 0) ? 1u : 0u);
          tc::mma_commit(&bar[B_EMPTY + slot]);
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
  } else {
    // ------------------------- queries, rotation, softmax and epilogue ---
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const PairInfo ri = pair_info(a, t, rq, m);
    const uint32_t lt = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    const int sink = a.sink, window = a.window;
    const uint16_t* qrow = ri.p >= 0 ? a.q + (ri.frow * a.H + ri.head) * DK : nullptr;
    // this lane's query: nope -> tensor memory (column c = dims 2c, 2c + 1),
    // rope kept in registers for the rotation of each segment
    uint32_t rope_raw[16];
    {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t w[32];
        if (qrow) {
          const uint4* s4 = reinterpret_cast<const uint4*>(qrow) + 8 * h;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 v = __ldg(s4 + u);
            w[4 * u] = v.x;
            w[4 * u + 1] = v.y;
            w[4 * u + 2] = v.z;
            w[4 * u + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) w[u] = 0;
        }
        tc::tmem_st32(lt + T_Q + 32 * h, w);
      }
      if (qrow) {
        const uint4* s4 = reinterpret_cast<const uint4*>(qrow + DN);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 v = __ldg(s4 + u);
          rope_raw[4 * u] = v.x;
          rope_raw[4 * u + 1] = v.y;
          rope_raw[4 * u + 2] = v.z;
          rope_raw[4 * u + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int u = 0; u < 16; ++u) rope_raw[u] = 0;
      }
    }
    KeyTile kt{0, 0, 0, -1};
    bool have = next_key_tile<TNK>(kt, segs, nseg, 0, r0hi, r1lo, r1hi);
    if (have) put_rope(lt, rope_raw, a.rope_cs + static_cast<int64_t>(rq.seg_first + kt.j) * DR);
    tc::tmem_wait_st();
    tc::tc_fence_before();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&bar[B_SFREE]);
    float m_run = -INFINITY, l_run = 0.f;
    int j = 0;
    bool ok = true;
    while (ok && have) {
      KeyTile nx = kt;
      const bool have_next = next_key_tile<TNK>(nx, segs, nseg, 0, r0hi, r1lo, r1hi);
      ok = __all_sync(0xffffffffu, wait_bar(c, B_SFULL, j & 1));
      if (!ok) break;
      tc::tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tc::tmem_ld32(lt + T_S + 32 * q4, s[q4]);
      tc::tmem_wait_ld();
      // S_j is complete, so no score MMA reads q_rope' any more: rotate the
      // query for the next segment before the next score MMAs are issued
      if (have_next && nx.j != kt.j) {
        put_rope(lt, rope_raw, a.rope_cs + static_cast<int64_t>(rq.seg_first + nx.j) * DR);
        tc::tmem_wait_st();
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[B_SFREE]);

      // scores are scaled inside the exponent: x = s * scale * log2(e)
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
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int key = kt.k0 + 32 * q4 + i;
            bool vis = key < kt.k1 && key <= p;
            if (!ri.glob) vis = vis && (key < sink || key >= p - window);
            const float x = vis ? __uint_as_float(s[q4][i]) : -INFINITY;
            s[q4][i] = __float_as_uint(x);
            mx4[i & 3] = fmaxf(mx4[i & 3], x);
          }
        }
      }
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
      bool need = false;
      float alpha = 1.f;
      if (mx > m_run + 8.f) {  // lazy rescale: only when the max grows by more than 2^8
        if (m_run != -INFINITY) {
          need = true;
          alpha = fast_exp2(m_run - mx);
        }
        m_run = mx;
      }
      const float nb = (m_run == -INFINITY) ? 0.f : -m_run;
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};
      // P in place: keys 2w, 2w + 1 in word w = 16 q4 + i of s[q4 >> 1]
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
      l_run = l_run * alpha + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
      // the previous P.V must be done before P and O are touched
      if (j >= 1) ok = __all_sync(0xffffffffu, wait_bar(c, B_ODONE, (j - 1) & 1));
      if (!ok) break;
      tc::tc_fence_after();
      tc::tmem_st32(lt + T_P, s[0]);
      tc::tmem_st32(lt + T_P + 32, s[1]);
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int q8 = 0; q8 < DV / 32; ++q8) {
          uint32_t o[32];
          tc::tmem_ld32(lt + T_O + 32 * q8, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tc::tmem_st32(lt + T_O + 32 * q8, o);
        }
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[B_PREADY]);
      ++j;
      kt = nx;
      have = have_next;
    }
    // ---- epilogue ----
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(c, B_FINAL, 0));
    tc::tc_fence_after();
    if (ok) {
      const bool st = ri.p >= 0 && l_run > 0.f;
      const float inv = st ? 1.f / l_run : 0.f;
      uint16_t* dst = st ? a.out + (ri.frow * a.H + ri.head) * DV : nullptr;
#pragma unroll 1
      for (int q8 = 0; q8 < DV / 32; ++q8) {
        uint32_t o[32];
        tc::tmem_ld32(lt + T_O + 32 * q8, o);
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
      if (st) a.lse[ri.frow * a.H + ri.head] = m_run * 0.6931471805599453f + logf(l_run);
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

cudaError_t launch_dense_tcs(const rk_seg_attn_plan_s& p, const KernelArgs& a, cudaStream_t s) {
  (void)p;
  cudaError_t e = cudaFuncSetAttribute(dense_tcs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  dense_tcs_kernel<<<static_cast<unsigned>(a.num_tiles), THREADS, SMEM_BYTES, s>>>(a);
  return cudaGetLastError();
}

}  // namespace rk
