// Short tile pairs on the SMs that the 4-CTA clusters leave free (tcgen05
// cta_group::2 + TMEM + TMA).
//
// SMs that do not divide into 4-CTA clusters stay idle while the 4-CTA
// prefill kernel runs (on a 152-SM GB300, 36 clusters hold 144 SMs).  This
// persistent kernel runs one CTA pair on each free SM pair, launched right
// after the 4-CTA kernel on a second stream, and takes tile pairs from the
// back of the same work queue while the 4-CTA clusters take them from the
// front: the plan orders pairs longest first, so it takes the shortest ones
// (Local tiles of protected rows, the first rows' Global tiles), and one
// 64-bit counter holds both ends, so every pair is taken exactly once.  It
// takes pairs only from the list's short tail (at most kSideMaxTiles key
// tiles each), so that a pair it starts late cannot lengthen the forward by
// much; if its CTAs find no free SMs they start after the 4-CTA kernel and
// find the queue empty.
//
// A CTA pair holds its two tiles' queries in shared memory (rank r: tile r's
// 128 lanes x the nope dims, loaded once per pair) and computes the output
// one half of d_v per pass over the keys, so the scores are computed twice.
// The arithmetic is the 4-CTA kernel's step for step, so that a pair's
// outputs do not depend on which kernel took it: the score chain S = Q K^T
// (M = 256, N = 128: 64 keys from each CTA's shared memory) takes the rope
// chunk's q_rope' hi and lo parts first and then the nope chunks in order,
// the query turning by -delta at each segment of the key walk (RedKnot-MLA
// paper, RoPE-orthogonality paragraph); the online softmax is the shared
// one; O += P V runs per 16 keys in key order after the rescale; the
// epilogue divides by the same running sum.  Two instantiations, as for the
// 4-CTA kernel: (d_nope, d_rope) = (512, 64) with V = c_nope, and (448, 64)
// with V = the whole latent row, whose rope columns (the last 64 of the
// second half) turn into each new segment's frame at a switch and get the
// output phase restored in the epilogue (RedKnot-MLA paper: R^-1 in the
// head-partition paragraph) by the 4-CTA kernel's own helpers.
// Tensor memory per CTA: O (256 columns) | S (128) | P (64) | q_rope' hi
// (32) | lo (32).  Every wait is bounded in time; on expiry the CTA records
// RK_ERR_DEVICE_TIMEOUT, every CTA of both kernels stops, the leader waits
// (bounded) for the pair's copies in flight, and tensor memory is released
// after the pair's MMA pipe has drained.

#include <algorithm>

#include "tc_tile.cuh"

namespace rk {
namespace {

using tt::Ctx;
using tt::drain_bar;
using tt::wait_bar;

constexpr int TNK = 128;
constexpr uint32_t CHUNK = 16384;  // 128 rows x 64 bf16
constexpr uint32_t HCHUNK = 8192;  // 64 rows x 64 bf16
constexpr int RING = 3;
constexpr uint32_t SLOT = 2 * CHUNK;
constexpr int THREADS = 192;

constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_RING = 8 * CHUNK;
constexpr uint32_t OFF_BAR = OFF_RING + RING * SLOT;
enum {
  B_FULL = 0,
  B_EMPTY = RING,
  B_QFULL = 2 * RING,  // one phase per pair
  B_QEMPTY,            // the pair's last score MMAs are done (one phase per pair)
  B_SFULL,
  B_SFREE,             // per lane of both CTAs: one arrival per pass, then one per tile
  B_PREADY,            // per lane of both CTAs: one arrival per tile
  B_ODONE,
  B_FINAL,             // one phase per pass
  B_SFINAL,            // every MMA of the launch is done (teardown)
  NBAR
};
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");

constexpr uint32_t T_O = 0, T_S = 256, T_P = 384, T_RH = 448, T_RL = 480;

// segment maps (kSegMaps per segment)
constexpr int MAP_V = 0;   // 128 rows x 2 chunks
constexpr int MAP_K4 = 2;  // 64 rows x 4 chunks
constexpr int MAP_R = 3;   // 64 rows x 1 chunk

// the side kernel's rings follow the 4-CTA clusters' rings in the queue
constexpr int RING_FIRST = kQueueClusters;

// The key walk of pair P (both tiles' key ranges) over request rq's segments.
__device__ __forceinline__ bool next_tile(KeyTile& kt, const TcPair& P, const DevSeg* segs,
                                          int nseg) {
  return next_key_tile<TNK>(kt, segs, nseg, 0, P.sink_hi, P.win_lo, P.key_hi,
                            static_cast<uint32_t>(P.skip));
}

template <int NCH, bool VROPE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    dense_side_kernel(const KernelArgs a, const __grid_constant__ tt::QMaps qm) {
  constexpr int DK = 64 * (NCH + 1);  // latent row: NCH nope chunks + the rope chunk
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  const Ctx c{bar, reinterpret_cast<volatile uint32_t*>(misc + 1), a.status};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = tc::cluster_ctarank();
  const int npairs = a.num_tc_pairs;
  // the leader's barrier i as a shared::cluster address
  auto lbar = [&](int i) { return tc::mapa_shared(smem_u32(&bar[i]), 0); };

  if (tid == 0) {
    for (int i = 0; i < RING; ++i) {
      tc::mbar_init(&bar[B_FULL + i], 1);
      tc::mbar_init(&bar[B_EMPTY + i], 1);
    }
    tc::mbar_init(&bar[B_QFULL], 1);
    tc::mbar_init(&bar[B_QEMPTY], 1);
    tc::mbar_init(&bar[B_SFULL], 1);
    tc::mbar_init(&bar[B_SFREE], 2 * 128);
    tc::mbar_init(&bar[B_PREADY], 2 * 128);
    tc::mbar_init(&bar[B_ODONE], 1);
    tc::mbar_init(&bar[B_FINAL], 1);
    tc::mbar_init(&bar[B_SFINAL], 1);
    misc[1] = 0;
    misc[3] = 0;  // rank 0: pairs whose outputs its lanes have written
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
      uint32_t cnt = 0, qloads = 0;
      bool ok = true;
      for (int item = 0; ok; ++item) {
        int idx;
        if (rank == 0) {
          // claim item `item` from the back of the list: its ring entry last
          // held item - kQueueRing, which every role has read once the lanes
          // (the last stage) have finished item - 48
          if (item >= 48) ok = tt::wait_count(c, &misc[3], static_cast<uint32_t>(item - 47));
          if (!ok) break;
          const unsigned long long old = atomicAdd(a.wq, 1ull << 32);
          const uint32_t front = static_cast<uint32_t>(old);
          const uint32_t back = static_cast<uint32_t>(old >> 32);
          const bool got = back < static_cast<uint32_t>(a.num_side_pairs) &&
                           static_cast<uint64_t>(front) + back < static_cast<uint64_t>(npairs);
          idx = got ? npairs - 1 - static_cast<int>(back) : -1;
          tc::st_release_gpu_u64(tt::queue_ring<2, RING_FIRST>(a.wq) + (item & (kQueueRing - 1)),
                                 (static_cast<unsigned long long>(item + 1) << 32) |
                                     static_cast<uint32_t>(idx));
        } else {
          idx = tt::claimed<2, RING_FIRST>(c, a.wq, item, npairs);
        }
        if (idx < 0) break;
        const TcPair& P = a.tc_pairs[idx];
        const TcTile t = P.t[rank];
        const DevReq rq = a.reqs[t.req];
        const DevSeg* segs = a.segs + rq.seg_first;
        const int nseg = rq.seg_count;
        // the queries: the buffer is free once the previous pair's last
        // score MMAs are done
        if (item > 0) ok = wait_bar(c, B_QEMPTY, (item - 1) & 1);
        if (!ok) break;
        // the leader's QFULL counts both CTAs' query bytes
        if (rank == 0) tc::mbar_arrive_expect_tx(&bar[B_QFULL], 2 * NCH * CHUNK);
        tt::load_q_tile<true, NCH>(a, qm, t, rq, smem_u32(sm + OFF_Q), lbar(B_QFULL));
        ++qloads;
        // one box per slot use; the leader arms its FULL barrier with both
        // CTAs' bytes, and both CTAs' copies complete on it
        auto load = [&](const KeyTile& kt, int map, int row_off, int z, uint32_t bytes) {
          const int slot = cnt % RING;
          const uint32_t ph = (cnt / RING) & 1;
          if (!wait_bar(c, B_EMPTY + slot, ph ^ 1)) return false;
          if (rank == 0) tc::mbar_arrive_expect_tx(&bar[B_FULL + slot], 2 * bytes);
          tc::tma_load_3d_2sm(smem_u32(sm + OFF_RING + slot * SLOT),
                              a.segmaps + kSegMaps * (rq.seg_first + kt.j) + map,
                              lbar(B_FULL + slot), 0, kt.k0 - segs[kt.j].delta + row_off, z);
          ++cnt;
          return true;
        };
        const int koff = 64 * static_cast<int>(rank);
        for (int half = 0; half < 2 && ok; ++half) {
          // per key tile: the rope chunk, nope chunks 0-3 and 4-7 of this
          // CTA's 64 keys (with NCH = 7 the second box's last chunk is the
          // rope chunk, unused), then this CTA's two value chunks of the
          // previous tile (the half's 256 columns: 128 from each CTA)
          KeyTile cur{0, 0, 0, -1}, prev{0, 0, 0, -1};
          bool have = next_tile(cur, P, segs, nseg);
          bool has_prev = false;
          while (ok && (have || has_prev)) {
            if (have) {
              ok = load(cur, MAP_R, koff, NCH, HCHUNK);
              if (ok) ok = load(cur, MAP_K4, koff, 0, 4 * HCHUNK);
              if (ok) ok = load(cur, MAP_K4, koff, 4, 4 * HCHUNK);
            }
            if (has_prev && ok)
              ok = load(prev, MAP_V, 0, 4 * half + 2 * static_cast<int>(rank), 2 * CHUNK);
            prev = cur;
            has_prev = have;
            if (have) have = next_tile(cur, P, segs, nseg);
          }
        }
      }
      // the pair's copies in flight land before either CTA may exit (the
      // teardown cluster barrier holds rank 1 until the leader gets here)
      if (rank == 0) {
        if (qloads) drain_bar(c, B_QFULL, (qloads - 1) & 1);
        for (uint32_t k = (cnt > RING ? cnt - RING : 0); k < cnt; ++k)
          drain_bar(c, B_FULL + k % RING, (k / RING) & 1);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------- MMA issuer (leader only) ---
    if (lane == 0 && rank == 0) {
      const uint32_t idS = tc::idesc_bf16(256, 128, false, false);
      const uint32_t idPV = tc::idesc_bf16(256, 256, false, true);
      const uint32_t qa = smem_u32(sm + OFF_Q), ra = smem_u32(sm + OFF_RING);
      uint32_t cnt = 0, sfree_ph = 0, pv = 0;
      bool ok = true;
      for (int item = 0; ok; ++item) {
        const int idx = tt::claimed<2, RING_FIRST>(c, a.wq, item, npairs);
        if (idx < 0) break;
        const TcPair& P = a.tc_pairs[idx];
        const DevReq rq = a.reqs[P.t[0].req];
        const DevSeg* segs = a.segs + rq.seg_first;
        const int nseg = rq.seg_count;
        ok = wait_bar(c, B_QFULL, item & 1);
        if (!ok) break;
        tc::tc_fence_after();
        bool q_released = false;
        for (int half = 0; half < 2 && ok; ++half) {
          KeyTile cur{0, 0, 0, -1};
          bool have = next_tile(cur, P, segs, nseg);
          bool has_prev = false, first = true;
          while (ok && (have || has_prev)) {
            KeyTile nx = cur;
            const bool have_next = have && next_tile(nx, P, segs, nseg);
            if (have) {
              // the lanes have read the previous S (and written the rotated
              // q_rope' for this tile's segment)
              ok = wait_bar<true>(c, B_SFREE, sfree_ph & 1);
              ++sfree_ph;
              if (!ok) break;
              tc::tc_fence_after();
              const uint32_t ts = tbase + T_S;
              // the rope chunk: A = q_rope' hi and lo from tensor memory
              int slot = cnt % RING;
              ok = wait_bar(c, B_FULL + slot, (cnt / RING) & 1);
              if (!ok) break;
              tc::tc_fence_after();
              uint32_t base = ra + slot * SLOT;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t bd = tc::sdesc_sw128(base + 32 * k, 16, 1024);
                tc::mma_ts_2sm(ts, tbase + T_RH + 8 * k, bd, idS, k != 0);
                tc::mma_ts_2sm(ts, tbase + T_RL + 8 * k, bd, idS, 1);
              }
              tc::mma_commit_2sm(&bar[B_EMPTY + slot], 0x3);
              ++cnt;
              // the nope chunks: A = Q from shared memory, B = K[64 keys of
              // each CTA x 16 dims]
              for (int b = 0; b < 2 && ok; ++b) {
                slot = cnt % RING;
                ok = wait_bar(c, B_FULL + slot, (cnt / RING) & 1);
                if (!ok) break;
                tc::tc_fence_after();
                base = ra + slot * SLOT;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                  const int cc = 4 * b + ch;
                  if (cc >= NCH) break;
#pragma unroll
                  for (int k = 0; k < 4; ++k)
                    tc::mma_ss_2sm(ts, tc::sdesc_sw128(qa + cc * CHUNK + 32 * k, 16, 1024),
                                   tc::sdesc_sw128(base + ch * HCHUNK + 32 * k, 16, 1024), idS, 1);
                }
                tc::mma_commit_2sm(&bar[B_EMPTY + slot], 0x3);
                ++cnt;
              }
              if (!ok) break;
              tc::mma_commit_2sm(&bar[B_SFULL], 0x3);
              // the pair's last score MMAs: its queries may be replaced
              if (half == 1 && !have_next) {
                tc::mma_commit_2sm(&bar[B_QEMPTY], 0x3);
                q_released = true;
              }
            }
            if (has_prev) {
              ok = wait_bar<true>(c, B_PREADY, pv & 1);
              if (!ok) break;
              tc::tc_fence_after();
              const int slot = cnt % RING;
              ok = wait_bar(c, B_FULL + slot, (cnt / RING) & 1);
              if (!ok) break;
              tc::tc_fence_after();
              const uint32_t base = ra + slot * SLOT;
              // B = V[16 keys x 256 columns]: 128 columns per CTA, as two
              // 64-column chunks 16 KB apart (LBO); the pass's first output
              // MMA starts the accumulator afresh
#pragma unroll
              for (int k = 0; k < 8; ++k)
                tc::mma_ts_2sm(tbase + T_O, tbase + T_P + 8 * k,
                               tc::sdesc_sw128(base + 2048 * k, CHUNK, 1024), idPV,
                               (!first || k > 0) ? 1u : 0u);
              tc::mma_commit_2sm(&bar[B_EMPTY + slot], 0x3);
              ++cnt;
              tc::mma_commit_2sm(&bar[B_ODONE], 0x3);
              ++pv;
              first = false;
            }
            has_prev = have;
            if (have) {
              cur = nx;
              have = have_next;
            }
          }
          if (!ok) break;
          tc::mma_commit_2sm(&bar[B_FINAL], 0x3);  // one phase per pass
          // the lanes' release after the pass's last S is not waited for: the
          // next pass's first S waits for their release after its q_rope'
          ++sfree_ph;
        }
        if (ok && !q_released) tc::mma_commit_2sm(&bar[B_QEMPTY], 0x3);
      }
      tc::mma_commit_2sm(&bar[B_SFINAL], 0x3);  // the pipe is empty before teardown
    }
  } else {
    // ---------------------------------- softmax, rotation and epilogue ---
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const uint32_t lt = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    const int sink = a.sink, window = a.window;
    const uint32_t sfree_l = lbar(B_SFREE), pready_l = lbar(B_PREADY);
    int j = 0;            // tiles of every pass so far
    uint32_t passes = 0;
    bool ok = true;
    for (int item = 0; ok; ++item) {
      const int idx = tt::claimed<2, RING_FIRST>(c, a.wq, item, npairs);
      if (idx < 0) break;
      const TcPair& P = a.tc_pairs[idx];
      const TcTile t = P.t[rank];
      const DevReq rq = a.reqs[t.req];
      const DevSeg* segs = a.segs + rq.seg_first;
      const int nseg = rq.seg_count;
      const tt::RowInfo ri = tt::row_info(a, t, rq, m);
      const uint16_t* qrope = ri.p >= 0 ? a.q + (ri.frow * a.H + ri.head) * DK + 64 * NCH : nullptr;
      for (int half = 0; half < 2 && ok; ++half) {
        KeyTile kt{0, 0, 0, -1};
        bool have = next_tile(kt, P, segs, nseg);
        // q_rope' of the first segment (every score MMA of the previous pass
        // is done: its last S has been read), then the pass's first release
        tt::write_rope(lt, T_RH, T_RL, qrope,
                       a.rope_cs + static_cast<int64_t>(rq.seg_first + kt.j) * 64);
        tc::tc_fence_before();
        tc::mbar_arrive_cluster(sfree_l);
        float m_run = -INFINITY, l_run = 0.f;
        // rotary value: the segment whose canonical frame the output's rope
        // columns are in (value columns 448..511: this CTA pair's columns
        // 192..255 in the second half)
        int seg_frame = kt.j;
        while (ok && have) {
          KeyTile nx = kt;
          const bool have_next = next_tile(nx, P, segs, nseg);
          ok = __all_sync(0xffffffffu, wait_bar(c, B_SFULL, j & 1));
          if (!ok) break;
          tc::tc_fence_after();
          // S_j is complete, so no score MMA still reads the rotated q_rope
          if (have_next && nx.j != kt.j)
            tt::write_rope(lt, T_RH, T_RL, qrope,
                           a.rope_cs + static_cast<int64_t>(rq.seg_first + nx.j) * 64);
          uint32_t s[4][32];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) tc::tmem_ld32(lt + T_S + 32 * q4, s[q4]);
          tc::tmem_wait_ld();
          tc::tc_fence_before();
          tc::mbar_arrive_cluster(sfree_l);
          // scores are scaled inside the exponent: x = s * scale * log2(e)
          const float alpha = tt::softmax_tile(s, kt, ri, sink, window, sl2, m_run, l_run);
          // the previous P.V must be done before P and O are touched
          if (j >= 1) ok = __all_sync(0xffffffffu, wait_bar(c, B_ODONE, (j - 1) & 1));
          if (!ok) break;
          tc::tc_fence_after();
          tc::tmem_st32(lt + T_P, s[0]);
          tc::tmem_st32(lt + T_P + 32, s[1]);
          const bool scale = __any_sync(0xffffffffu, alpha != 1.f);
          // a new segment: R(delta_frame - delta_next) moves the rope columns
          // into the next segment's canonical frame (after the rescale, as
          // the 4-CTA kernel does)
          const bool turn = VROPE && half == 1 && kt.j != seg_frame;
          if (scale || turn) {
            const float4* ca =
                reinterpret_cast<const float4*>(a.rope_cs + int64_t(rq.seg_first + seg_frame) * 64);
            const float4* cb =
                reinterpret_cast<const float4*>(a.rope_cs + int64_t(rq.seg_first + kt.j) * 64);
#pragma unroll 1
            for (int q8 = scale ? 0 : 6; q8 < 8; ++q8) {
              uint32_t o[32];
              tc::tmem_ld32(lt + T_O + 32 * q8, o);
              tc::tmem_wait_ld();
              if (scale) {
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              }
              if (turn && q8 >= 6) tt::turn16(o, ca, cb, 16 * (q8 - 6));
              tc::tmem_st32(lt + T_O + 32 * q8, o);
            }
          }
          seg_frame = kt.j;
          tc::tmem_wait_st();
          tc::tc_fence_before();
          tc::mbar_arrive_cluster(pready_l);
          ++j;
          kt = nx;
          have = have_next;
        }
        // ---- epilogue of this half ----
        if (ok) ok = __all_sync(0xffffffffu, wait_bar(c, B_FINAL, passes & 1));
        ++passes;
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
            if (VROPE && st && half == 1 && q8 >= 6) {
              // rotary value: R(delta_frame - p) restores the last segment's
              // output phase and applies the inverse output RoPE at the row's
              // position p (cos / sin of p theta from the two-level table)
              const float4* ca =
                  reinterpret_cast<const float4*>(a.rope_cs + int64_t(rq.seg_first + seg_frame) * 64);
              const float4* ph = reinterpret_cast<const float4*>(a.pos_cs_hi + int64_t(ri.p >> 8) * 64);
              const float4* pl = reinterpret_cast<const float4*>(a.pos_cs_lo + int64_t(ri.p & 255) * 64);
              tt::restore16(o, ca, ph, pl, 16 * (q8 - 6));
            }
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
          if (st && half == 0)
            a.lse[ri.frow * a.H + ri.head] = tt::lse_of(m_run, l_run);
        }
      }
      // rank 0 reports the pairs it has finished: the claimer reuses a ring
      // entry only once these are 16 items past its last reader
      if (ok && rank == 0 && m == 0)
        tc::st_release_cluster_u32(tc::mapa_shared(smem_u32(&misc[3]), 0),
                                   static_cast<uint32_t>(item + 1));
    }
  }

  // ------------------------------------------------------------ teardown --
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) drain_bar(c, B_SFINAL, 0);  // the pair's MMA pipe is empty
  __syncthreads();
  tc::cluster_sync();  // neither CTA leaves while the other may still use its memory
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc_2sm(tbase, 512);
  }
}

}  // namespace

cudaError_t prepare_dense_side() {
  cudaError_t e = cudaFuncSetAttribute(dense_side_kernel<8, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(dense_side_kernel<7, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(SMEM_BYTES));
}

cudaError_t launch_dense_side(const rk_seg_attn_plan_s& p, const KernelArgs& a, const void* q,
                              int64_t tc4_clusters, cudaStream_t s) {
  const bool vr = p.v_rope;
  if (p.d_rope != 64 || p.d_nope != (vr ? 448 : 512) || a.num_side_pairs <= 0 || !a.wq)
    return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // one CTA pair per free SM pair (each CTA fills an SM's shared memory)
  const int64_t pairs = std::min<int64_t>(
      std::min<int64_t>((static_cast<int64_t>(sms) - 4 * tc4_clusters) / 2, kSideClusters),
      a.num_side_pairs);
  if (pairs <= 0) return cudaSuccess;
  tt::QMaps qm;
  e = tt::make_qmaps(p, a, q, qm);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(2 * pairs));
  if (vr)
    dense_side_kernel<7, true><<<grid, THREADS, SMEM_BYTES, s>>>(a, qm);
  else
    dense_side_kernel<8, false><<<grid, THREADS, SMEM_BYTES, s>>>(a, qm);
  return cudaGetLastError();
}

}  // namespace rk
