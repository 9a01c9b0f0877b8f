// Prefill-style tiles on CTA pairs (tcgen05 cta_group::2 + TMEM + TMA).
//
// A cluster of two CTAs takes two 128-pair tiles of one request (rank r
// holds tile r) and one half of d_v, and walks the union of the two tiles'
// key ranges.  The pair shares every latent byte it streams: for a key tile
// of 128 keys each CTA loads only its 64 keys of the score operand (two
// 32 KB boxes of 64 keys x 4 chunks and an 8 KB box of the rope chunk) and
// its two of this half's four V-column chunks (one 32 KB box of 128 keys x
// 2 chunks), so a CTA streams 104 KB per key tile instead of 224 KB.  One
// thread of rank 0 issues the MMAs for both CTAs:
//   S  = Q K^T   M = 256 (128 rows per CTA), N = 128 keys (64 from each
//                CTA's shared memory), K: 8 nope chunks with A = Q from
//                shared memory, the rope chunk with A = q_rope' hi and lo
//                from each CTA's tensor memory;
//   O += P V     M = 256, N = 256 output columns (128 from each CTA's
//                shared memory, MN-major), A = P from each CTA's TMEM.
// Tensor memory per CTA: O (256) | S (128) | P (64) | q_rope' hi (32) | lo (32).
//
// Each CTA's softmax warpgroup works on its own 128 rows as in the one-CTA
// tcgen05 kernel: the query turns by -delta at each segment of the key walk
// and the running max / sum / output carry across segments as a log-sum-exp
// merge (RedKnot-MLA paper, RoPE-orthogonality paragraph); Global rows see
// k <= p and Local rows sink u [p - w, p] (RedKnot blog, "Insight 1").  Its
// arrivals go to the leader's barriers; the leader's MMA completions are
// multicast to both CTAs, and rank 1's TMA loads complete on the leader's
// barriers.  Every wait is bounded in time; on expiry the CTA records
// RK_ERR_DEVICE_TIMEOUT, the other CTAs see the status word and stop, the
// leader waits (bounded) for the pair's copies in flight, and tensor memory
// is released after the pair's MMA pipe has drained.

#include "tc_tile.cuh"

namespace rk {
namespace {

constexpr int TNK = 128;
constexpr uint32_t CHUNK = 16384;          // 128 rows x 64 bf16
constexpr uint32_t HCHUNK = 8192;          // 64 rows x 64 bf16
constexpr int RING = 3;
constexpr uint32_t SLOT = 2 * CHUNK;
constexpr int THREADS = 192;

constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_RING = 8 * CHUNK;
constexpr uint32_t OFF_BAR = OFF_RING + RING * SLOT;
enum { B_FULL = 0, B_EMPTY = RING, B_QFULL = 2 * RING, B_SFULL, B_SFREE, B_PREADY, B_ODONE, B_FINAL, NBAR };
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;

constexpr uint32_t T_O = 0, T_S = 256, T_P = 384, T_RH = 448, T_RL = 480;

// segment maps, 4 per segment
constexpr int MAP_V = 0;     // 128 rows x 2 chunks
constexpr int MAP_K4 = 2;    // 64 rows x 4 chunks
constexpr int MAP_R = 3;     // 64 rows x 1 chunk

using tt::Ctx;
using tt::drain_bar;
using tt::wait_bar;


__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    dense_tc2_kernel(const KernelArgs a, const __grid_constant__ tt::QMaps qm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  const Ctx c{bar, reinterpret_cast<volatile uint32_t*>(misc + 1), a.status};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = tc::cluster_ctarank();
  const int half = (blockIdx.x >> 1) & 1;
  const TcPair& P = a.tc_pairs[blockIdx.x >> 2];
  const TcTile t = P.t[rank];
  const DevReq rq = a.reqs[t.req];
  const DevSeg* segs = a.segs + rq.seg_first;
  const int nseg = rq.seg_count;
  const int r0hi = P.sink_hi, r1lo = P.win_lo, r1hi = P.key_hi;
  const uint32_t skip = static_cast<uint32_t>(P.skip);
  // the leader's barrier i as a shared::cluster address
  auto lbar = [&](int i) { return tc::mapa_shared(smem_u32(&bar[i]), 0); };

  if (tid == 0) {
    for (int i = 0; i < RING; ++i) {
      tc::mbar_init(&bar[B_FULL + i], 1);
      tc::mbar_init(&bar[B_EMPTY + i], 1);
    }
    tc::mbar_init(&bar[B_QFULL], 1);
    tc::mbar_init(&bar[B_SFULL], 1);
    tc::mbar_init(&bar[B_SFREE], 2 * 128);
    tc::mbar_init(&bar[B_PREADY], 2 * 128);
    tc::mbar_init(&bar[B_ODONE], 1);
    tc::mbar_init(&bar[B_FINAL], 1);
    misc[1] = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc_2sm(misc, 512);
    tc::tmem_relinquish_2sm();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();  // the peer's barriers are initialised before any remote arrive
  tc::tc_fence_after();
  const uint32_t tbase = misc[0];

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      // the leader's QFULL counts both CTAs' Q bytes
      if (rank == 0) tc::mbar_arrive_expect_tx(&bar[B_QFULL], 2 * 8 * CHUNK);
      tt::load_q_tile<true>(a, qm, t, rq, smem_u32(sm + OFF_Q), lbar(B_QFULL));
      uint32_t cnt = 0;
      bool ok = true;
      // one box per slot use; the leader arms its FULL barrier with both
      // CTAs' bytes, and both CTAs' copies complete on it
      auto load = [&](const KeyTile& kt, int map, int row_off, int z, uint32_t bytes) {
        const int slot = cnt % RING;
        const uint32_t ph = (cnt / RING) & 1;
        if (!wait_bar(c, B_EMPTY + slot, ph ^ 1)) return false;
        if (rank == 0) tc::mbar_arrive_expect_tx(&bar[B_FULL + slot], 2 * bytes);
        tc::tma_load_3d_2sm(smem_u32(sm + OFF_RING + slot * SLOT),
                            a.segmaps + kSegMaps * (rq.seg_first + kt.j) + map, lbar(B_FULL + slot), 0,
                            kt.k0 - segs[kt.j].delta + row_off, z);
        ++cnt;
        return true;
      };
      KeyTile cur{0, 0, 0, -1}, prev{0, 0, 0, -1};
      bool have = next_key_tile<TNK>(cur, segs, nseg, 0, r0hi, r1lo, r1hi, skip);
      bool has_prev = false;
      const int koff = 64 * static_cast<int>(rank);
      while (ok && (have || has_prev)) {
        if (have) {
          ok = load(cur, MAP_K4, koff, 0, 4 * HCHUNK);
          if (ok) ok = load(cur, MAP_K4, koff, 4, 4 * HCHUNK);
          if (ok) ok = load(cur, MAP_R, koff, 8, HCHUNK);
        }
        if (has_prev && ok)
          ok = load(prev, MAP_V, 0, 4 * half + 2 * static_cast<int>(rank), 2 * CHUNK);
        prev = cur;
        has_prev = have;
        if (have) have = next_key_tile<TNK>(cur, segs, nseg, 0, r0hi, r1lo, r1hi, skip);
      }
      // the pair's copies in flight land before either CTA may exit (the
      // teardown cluster barrier holds rank 1 until the leader gets here)
      if (rank == 0) {
        drain_bar(c, B_QFULL, 0);
        for (uint32_t k = (cnt > RING ? cnt - RING : 0); k < cnt; ++k)
          drain_bar(c, B_FULL + k % RING, (k / RING) & 1);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------- MMA issuer (leader only) ---
    if (lane == 0 && rank == 0) {
      bool ok = wait_bar(c, B_QFULL, 0);
      tc::tc_fence_after();
      const uint32_t idS = tc::idesc_bf16(256, 128, false, false);
      const uint32_t idPV = tc::idesc_bf16(256, 256, false, true);
      const uint32_t qa = smem_u32(sm + OFF_Q), ra = smem_u32(sm + OFF_RING);
      uint32_t cnt = 0;
      int j = 0, jprev = -1;
      KeyTile cur{0, 0, 0, -1};
      bool have = next_key_tile<TNK>(cur, segs, nseg, 0, r0hi, r1lo, r1hi, skip);
      bool has_prev = false;
      while (ok && (have || has_prev)) {
        if (have) {
          ok = wait_bar(c, B_SFREE, j & 1);
          if (!ok) break;
          tc::tc_fence_after();
          for (int b = 0; b < 3 && ok; ++b) {
            const int slot = cnt % RING;
            ok = wait_bar(c, B_FULL + slot, (cnt / RING) & 1);
            if (!ok) break;
            tc::tc_fence_after();
            const uint32_t base = ra + slot * SLOT;
            if (b < 2) {
              // B = K[64 keys of each CTA x 64 dims] of nope chunk 4b + ch
#pragma unroll
              for (int ch = 0; ch < 4; ++ch) {
                const int cc = 4 * b + ch;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  tc::mma_ss_2sm(tbase + T_S, tc::sdesc_sw128(qa + cc * CHUNK + 32 * k, 16, 1024),
                                 tc::sdesc_sw128(base + ch * HCHUNK + 32 * k, 16, 1024), idS,
                                 (cc | k) != 0);
              }
            } else {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t bd = tc::sdesc_sw128(base + 32 * k, 16, 1024);
                tc::mma_ts_2sm(tbase + T_S, tbase + T_RH + 8 * k, bd, idS, 1);
                tc::mma_ts_2sm(tbase + T_S, tbase + T_RL + 8 * k, bd, idS, 1);
              }
            }
            tc::mma_commit_2sm(&bar[B_EMPTY + slot], 0x3);
            ++cnt;
          }
          if (!ok) break;
          tc::mma_commit_2sm(&bar[B_SFULL], 0x3);
        }
        if (has_prev) {
          ok = wait_bar(c, B_PREADY, jprev & 1);
          if (!ok) break;
          tc::tc_fence_after();
          const int slot = cnt % RING;
          ok = wait_bar(c, B_FULL + slot, (cnt / RING) & 1);
          if (!ok) break;
          tc::tc_fence_after();
          const uint32_t base = ra + slot * SLOT;
          // B = V[16 keys x 256 columns]: 128 columns per CTA, as two 64-column
          // chunks 16 KB apart (LBO)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc::mma_ts_2sm(tbase + T_O, tbase + T_P + 8 * k,
                           tc::sdesc_sw128(base + 2048 * k, CHUNK, 1024), idPV,
                           (jprev > 0 || k > 0) ? 1u : 0u);
          tc::mma_commit_2sm(&bar[B_EMPTY + slot], 0x3);
          ++cnt;
          tc::mma_commit_2sm(&bar[B_ODONE], 0x3);
        }
        has_prev = have;
        jprev = j;
        if (have) {
          have = next_key_tile<TNK>(cur, segs, nseg, 0, r0hi, r1lo, r1hi, skip);
          ++j;
        }
      }
      tc::mma_commit_2sm(&bar[B_FINAL], 0x3);
    }
  } else {
    // ---------------------------------- softmax, rotation and epilogue ---
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const tt::RowInfo ri = tt::row_info(a, t, rq, m);
    const uint32_t lt = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    const int sink = a.sink, window = a.window;
    const uint16_t* qrope = ri.p >= 0 ? a.q + (ri.frow * a.H + ri.head) * 576 + 512 : nullptr;
    const uint32_t sfree_l = lbar(B_SFREE), pready_l = lbar(B_PREADY);
    KeyTile kt{0, 0, 0, -1};
    bool have = next_key_tile<TNK>(kt, segs, nseg, 0, r0hi, r1lo, r1hi, skip);
    // q_rope' of the first segment, then release the (empty) S buffer
    tt::write_rope(lt, T_RH, T_RL, qrope, a.rope_cs + static_cast<int64_t>(rq.seg_first + kt.j) * 64);
    tc::tc_fence_before();
    tc::mbar_arrive_cluster(sfree_l);
    float m_run = -INFINITY, l_run = 0.f;
    int j = 0;
    bool ok = true;
    while (ok && have) {
      KeyTile nx = kt;
      const bool have_next = next_key_tile<TNK>(nx, segs, nseg, 0, r0hi, r1lo, r1hi, skip);
      ok = __all_sync(0xffffffffu, wait_bar(c, B_SFULL, j & 1));
      if (!ok) break;
      tc::tc_fence_after();
      // S_j is complete, so no score MMA still reads the rotated q_rope
      if (have_next && nx.j != kt.j)
        tt::write_rope(lt, T_RH, T_RL, qrope, a.rope_cs + static_cast<int64_t>(rq.seg_first + nx.j) * 64);
      uint32_t s[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tc::tmem_ld32(lt + T_S + 32 * q4, s[q4]);
      tc::tmem_wait_ld();
      tc::tc_fence_before();
      tc::mbar_arrive_cluster(sfree_l);

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
      if (mx > m_run + 8.f) {
        if (m_run != -INFINITY) {
          need = true;
          alpha = fast_exp2(m_run - mx);
        }
        m_run = mx;
      }
      const float nb = (m_run == -INFINITY) ? 0.f : -m_run;
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};
      // P in place: pair i of column block q4 goes to word 16 * q4 + i
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
        for (int q8 = 0; q8 < 8; ++q8) {
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
      tc::mbar_arrive_cluster(pready_l);
      ++j;
      kt = nx;
      have = have_next;
    }
    // ---- epilogue ----
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(c, B_FINAL, 0));
    tc::tc_fence_after();
    if (ok) {
      const bool st = ri.store && l_run > 0.f;
      const float inv = st ? 1.f / l_run : 0.f;
      uint16_t* dst = st ? a.out + (ri.frow * a.H + ri.head) * 512 + 256 * half : nullptr;
#pragma unroll 1
      for (int q8 = 0; q8 < 8; ++q8) {
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
      if (st && half == 0) a.lse[ri.frow * a.H + ri.head] = m_run * 0.6931471805599453f + logf(l_run);
    }
  }

  // ------------------------------------------------------------ teardown --
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) drain_bar(c, B_FINAL, 0);  // the pair's MMA pipe is empty
  __syncthreads();
  tc::cluster_sync();  // neither CTA leaves while the other may still use its memory
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc_2sm(tbase, 512);
  }
}

}  // namespace

cudaError_t launch_dense_tc2(const rk_seg_attn_plan_s& p, const KernelArgs& a, const void* q,
                             cudaStream_t s) {
  tt::QMaps qm;
  cudaError_t e = tt::make_qmaps(p, a, q, qm);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(dense_tc2_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  const int64_t grid = 4 * static_cast<int64_t>(a.num_tc_pairs);
  dense_tc2_kernel<<<static_cast<unsigned>(grid), THREADS, SMEM_BYTES, s>>>(a, qm);
  return cudaGetLastError();
}

}  // namespace rk
