// Prefill-style tiles on 4-CTA clusters: the scores of two tiles on one CTA
// pair, their outputs on another (tcgen05 cta_group::2 + TMEM + TMA).
//
// Tensor memory cannot hold a tile's fp32 output over all of d_v (128 x 512
// columns) next to its scores, so a tile handled by one CTA pair per half
// of d_v computes S = Q K^T twice.  Here the work is split by role instead:
//
//   ranks 0, 1  "S pair": rank r holds tile r's queries, the nope part in
//               tensor memory (32 columns per 64 dims, A operand of the score
//               MMAs) and the rotated rope part in shared memory, and computes
//               S_j = Q K_j^T for both tiles with M = 256 MMAs (N = 128
//               keys: rank r streams keys 64r..64r+63 of every key tile as
//               one box of whole latent rows through a two-slot ring) into
//               one of two S buffers, runs the online softmax of its 128
//               lanes, stages P_j (bf16, two 16 KB halves in three rotating
//               slots of its shared memory) and bulk-copies each half into the
//               shared memory of rank r + 2; the per-lane record (rescale
//               factor, running sum) goes there by st.async.
//   ranks 2, 3  "O pair": rank 2 + r holds tile r's fp32 output for all 512
//               columns in tensor memory and computes O += P_j V_j with
//               M = 256, N = 2 x 256 MMAs (A = P_j from shared memory; rank
//               2 + r streams value chunks 4r..4r+3 of every key tile, 64 KB,
//               through a two-slot ring), rescales O when the record says
//               so, and stores the normalised output.
//
// Two instantiations: (d_nope, d_rope) = (512, 64) with V = c_nope, and
// (448, 64) with a value that carries a rotary part (V = the whole 512-wide
// latent row).  In the second the output's rope columns are kept in the
// canonical frame of the segment being walked: at a segment switch the O
// lanes turn them by R(delta_prev - delta_next), and the epilogue turns them
// by R(delta_last - p), which restores each segment's output phase and
// applies the inverse output RoPE at the row's position p (RedKnot-MLA
// paper: R^-1 in the head-partition paragraph, "restores the output phase"
// in the RoPE-orthogonality paragraph).
//
// Clusters are persistent: each walks a sequence of tile pairs (the plan's
// pairs, longest first, dealt out in rounds), with every ring, buffer and
// barrier phase carried from one pair to the next, so that one pair's output
// epilogue overlaps the next pair's query load on the score side.  Each
// latent byte is read once per pair, every MMA does useful work, and the
// score and output MMAs of a key tile run on different SMs at the same
// time.  The method is the one of the other prefill kernels: the query
// rotates by -delta at each segment of the key walk and the running max /
// sum / output carry across segments as a log-sum-exp merge (RedKnot-MLA
// paper, RoPE-orthogonality paragraph); Global rows see k <= p and Local
// rows sink u [p - w, p] (RedKnot blog, "Insight 1").  Every wait is bounded
// in time; on expiry the CTA records RK_ERR_DEVICE_TIMEOUT, every CTA of the
// launch stops, leaders wait (bounded) for their copies in flight, and
// tensor memory is released after each pair's MMA pipe has drained.

#include <algorithm>

#include "tc_tile.cuh"

namespace rk {
namespace {

using tt::Ctx;
using tt::drain_bar;
using tt::wait_bar;

constexpr int TNK = 128;                   // keys per key tile
constexpr uint32_t CHUNK = 16384;          // 128 rows x 64 bf16
constexpr uint32_t HCHUNK = 8192;          // 64 rows x 64 bf16
constexpr int THREADS = 256;   // warps 6 and 7: the rope writers of the score pair

// S pair: rotated q_rope hi and lo (K-major operands), three staging slots
// for P halves (64 keys x 128 lanes each), the key ring
constexpr uint32_t OFF_ROPE = 0;
constexpr uint32_t PBUF = 2 * CHUNK;       // 128 lanes x 128 keys bf16, two 64-key chunks
constexpr uint32_t RBUF = 128 * 8;         // (alpha, l) per lane, after P
constexpr uint32_t PSTRIDE = PBUF + 2048;  // 1024-aligned buffers
constexpr uint32_t OFF_STG = 2 * CHUNK;
constexpr int NSTG = 3;                    // staging slots; half k of the walk uses slot k % 3
constexpr int KRING = 2;
constexpr uint32_t KSLOT = 9 * HCHUNK;     // 64 keys x up to 9 chunks: one box per key tile
constexpr uint32_t OFF_KRING = OFF_STG + NSTG * CHUNK;
// O pair: two P + record buffers, the V ring (128 keys x 4 chunks per slot)
constexpr uint32_t OFF_P = 0;
constexpr int VRING = 2;
constexpr uint32_t VSLOT = 4 * CHUNK;
constexpr uint32_t OFF_VRING = OFF_P + 2 * PSTRIDE;
constexpr uint32_t OFF_BAR = OFF_KRING + KRING * KSLOT;
static_assert(OFF_KRING % 1024 == 0 && OFF_VRING % 1024 == 0, "operand alignment");
static_assert(OFF_VRING + VRING * VSLOT <= OFF_BAR, "O-pair layout");
static_assert(OFF_STG + 4 * 4096 <= OFF_KRING, "query transposition slices");
enum {
  B_KFULL = 0,
  B_KEMPTY = B_KFULL + KRING,
  B_SFULL = B_KEMPTY + KRING,  // 2: S buffer j & 1 written
  // SFREE, ROPE and PREADY take one arrival per lane warp of both CTAs of a
  // pair, made by lane 0 after the warp has synchronised
  B_SFREE = B_SFULL + 2,  // 2: S buffer read by both S CTAs' softmax lanes
  B_ROPE = B_SFREE + 2,   // rotated q_rope of the next segment written (one arrival
                          // per rope warp of both S CTAs)
  B_QREADY,               // queries in tensor memory (one arrival per lane warp)
  B_SWITCH,               // the rope MMAs of a segment's last tile are done (one phase
                          // per segment switch, so the rope warps wait on every phase)
  B_SFINAL,
  B_PEMPTY,             // 2 (S CTAs): P buffer consumed by the output MMAs
  B_VFULL = B_PEMPTY + 2,
  B_VEMPTY = B_VFULL + VRING,
  // 2 + 2 (O CTAs): P keys 0-63 copied in; P keys 64-127 and the records in
  B_PFULL0 = B_VEMPTY + VRING,
  B_PFULL1 = B_PFULL0 + 2,
  B_PREADY = B_PFULL1 + 2,     // 2: O rescaled where needed, P buffer ready for the MMAs
  B_ODONE = B_PREADY + 2,
  B_OFINAL,
  NBAR
};
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");

// tensor memory: S pair | O pair
constexpr uint32_t T_Q = 0, T_S = 256;
constexpr uint32_t T_O = 0;

// segment maps (kSegMaps per segment)
constexpr int MAP_K9 = 4;    // 64 rows x all d_k / 64 chunks
constexpr int MAP_V4 = 5;    // 128 rows x 4 chunks

// One tile pair of a cluster's walk, as seen by CTA rank r of a pair.
struct Item {
  TcTile t;
  DevReq rq;
  const DevSeg* segs;
  int nseg, r0hi, r1lo, r1hi;
  uint32_t skip;
};
__device__ __forceinline__ Item load_item(const KernelArgs& a, int idx, uint32_t r) {
  const TcPair& P = a.tc_pairs[idx];
  Item it;
  it.t = P.t[r];
  it.rq = a.reqs[it.t.req];
  it.segs = a.segs + it.rq.seg_first;
  it.nseg = it.rq.seg_count;
  it.r0hi = P.sink_hi;
  it.r1lo = P.win_lo;
  it.r1hi = P.key_hi;
  it.skip = static_cast<uint32_t>(P.skip);
  return it;
}
// Items are claimed dynamically: the score CTA of rank 0 (its TMA producer,
// which runs ahead of every other role) takes the next pair index from the
// front of the launch's counter (the plan orders pairs longest first; the
// side kernel takes pairs from the back) and publishes it in its cluster's
// ring as (k + 1) << 32 | index for item k of the walk; every other role
// reads the ring.  An index >= npairs (0xffffffff) ends the walk.
__device__ __forceinline__ unsigned long long* ring_of(unsigned long long* wq) {
  return tt::queue_ring<4, 0>(wq);
}
__device__ __forceinline__ bool next_tile(KeyTile& kt, const Item& I) {
  return next_key_tile<TNK>(kt, I.segs, I.nseg, 0, I.r0hi, I.r1lo, I.r1hi, I.skip);
}

template <int NCH, bool VROPE>
__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(THREADS, 1)
    dense_tc4_kernel(const KernelArgs a) {
  constexpr int DK = 64 * (NCH + 1);           // latent row: NCH nope chunks + the rope chunk
  constexpr uint32_t KBOX = (NCH + 1) * HCHUNK;  // one CTA's key box
  static_assert(KBOX <= KSLOT, "key slot");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  const Ctx c{bar, reinterpret_cast<volatile uint32_t*>(misc + 1), a.status};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = tc::cluster_ctarank();
  const bool spair = crank < 2;
  const uint32_t r = crank & 1;      // tile of the pair
  const int npairs = a.num_tc_pairs;
  auto cbar = [&](int i, uint32_t rank) { return tc::mapa_shared(smem_u32(&bar[i]), rank); };

  if (tid == 0) {
    for (int i = 0; i < KRING; ++i) {
      tc::mbar_init(&bar[B_KFULL + i], 1);
      tc::mbar_init(&bar[B_KEMPTY + i], 1);
    }
    for (int i = 0; i < VRING; ++i) {
      tc::mbar_init(&bar[B_VFULL + i], 1);
      tc::mbar_init(&bar[B_VEMPTY + i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bar[B_SFULL + b], 1);
      tc::mbar_init(&bar[B_SFREE + b], 2 * 4);
      tc::mbar_init(&bar[B_PEMPTY + b], 1);
      tc::mbar_init(&bar[B_PFULL0 + b], 1);
      tc::mbar_init(&bar[B_PFULL1 + b], 1);
      tc::mbar_init(&bar[B_PREADY + b], 2 * 4);
    }
    tc::mbar_init(&bar[B_ROPE], 2 * 2);
    tc::mbar_init(&bar[B_QREADY], 2 * 4);
    tc::mbar_init(&bar[B_SWITCH], 1);
    tc::mbar_init(&bar[B_SFINAL], 1);
    tc::mbar_init(&bar[B_ODONE], 1);
    tc::mbar_init(&bar[B_OFINAL], 1);
    misc[1] = 0;
    misc[2] = 0;  // S CTAs: P halves of the walk landed at the output CTA, in order
    misc[3] = 0;  // rank 0: items whose output the O lanes of rank 2 have written
    if (!spair)  // each P buffer expects one bulk copy per use; armed one use ahead
      for (int b = 0; b < 2; ++b) {
        tc::mbar_arrive_expect_tx(&bar[B_PFULL0 + b], CHUNK);
        tc::mbar_arrive_expect_tx(&bar[B_PFULL1 + b], CHUNK + RBUF);
      }
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc_2sm(misc, 512);
    tc::tmem_relinquish_2sm();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();  // every barrier of the cluster is initialised before any remote use
  tc::tc_fence_after();
  const uint32_t tbase = misc[0];

  if (spair) {
    if (warp == 0) {
      // ------------------------------------------- S pair: TMA producer --
      if (lane == 0) {
        uint32_t cnt = 0;
        bool ok = true;
        for (int item = 0; ok; ++item) {
          int idx;
          if (r == 0) {
            // claim item `item`: its ring entry last held item - kQueueRing,
            // which every role has read once the O lanes (the last stage)
            // have finished item - 48
            if (item >= 48) ok = wait_count(c, &misc[3], static_cast<uint32_t>(item - 47));
            if (!ok) break;
            // the next pair from the front of the list, unless the side
            // kernel has taken it from the back (it takes at most the
            // num_side_pairs shortest ones)
            const unsigned long long old = atomicAdd(a.wq, 1ull);
            const uint32_t front = static_cast<uint32_t>(old);
            const uint32_t back = static_cast<uint32_t>(old >> 32);
            const uint32_t taken = min(back, static_cast<uint32_t>(a.num_side_pairs));
            idx = static_cast<uint64_t>(front) + taken < static_cast<uint64_t>(npairs)
                      ? static_cast<int>(front) : -1;
            tc::st_release_gpu_u64(ring_of(a.wq) + (item & (kQueueRing - 1)),
                                   (static_cast<unsigned long long>(item + 1) << 32) |
                                       static_cast<uint32_t>(idx));
          } else {
            idx = tt::claimed<4, 0>(c, a.wq, item, a.num_tc_pairs);
          }
          if (idx < 0) break;
          const Item I = load_item(a, idx, r);
          // a Local tile's queries are whole rows (every head of one or two
          // rows): bring them into L2 while the lanes finish the previous item
          if (I.t.kind == 1 && !(I.t.pad & 1)) {
            const uint32_t rb = static_cast<uint32_t>(a.H) * DK * 2;
            const int nrow = a.H >= 128 ? 1 : 2;
            for (int rr = 0; rr < nrow; ++rr) {
              const int p = rr == 0 ? I.t.p0 : I.t.p1;
              if (p >= 0)
                tc::bulk_prefetch_l2(a.q + (I.rq.row_base + (p - I.rq.q_row_begin)) * a.H * DK, rb);
            }
          }
          KeyTile cur{0, 0, 0, -1};
          bool have = next_tile(cur, I);
          while (ok && have) {
            const int slot = cnt % KRING;
            ok = wait_bar(c, B_KEMPTY + slot, ((cnt / KRING) & 1) ^ 1);
            if (!ok) break;
            // the leader's barrier counts both CTAs' boxes
            if (r == 0) tc::mbar_arrive_expect_tx(&bar[B_KFULL + slot], 2 * KBOX);
            tc::tma_load_3d_2sm(smem_u32(sm + OFF_KRING + slot * KSLOT),
                                a.segmaps + kSegMaps * (I.rq.seg_first + cur.j) + MAP_K9,
                                cbar(B_KFULL + slot, 0), 0,
                                cur.k0 - I.segs[cur.j].delta + 64 * static_cast<int>(r), 0);
            ++cnt;
            have = next_tile(cur, I);
          }
        }
        // the pair's copies in flight land before either CTA may exit
        if (r == 0)
          for (uint32_t k = (cnt > KRING ? cnt - KRING : 0); k < cnt; ++k)
            drain_bar(c, B_KFULL + k % KRING, (k / KRING) & 1);
      }
    } else if (warp == 1) {
      // ------------------------------ S pair: MMA issuer (rank 0 only) --
      if (lane == 0 && r == 0) {
        const uint32_t idS = tc::idesc_bf16(256, 128, false, false);
        const uint32_t ropa = smem_u32(sm + OFF_ROPE), ka = smem_u32(sm + OFF_KRING);
        uint32_t rope_ev = 0, cnt = 0;
        int j = 0;
        bool ok = true;
        for (int item = 0; ok; ++item) {
          const int idx = tt::claimed<4, 0>(c, a.wq, item, a.num_tc_pairs);
          if (idx < 0) break;
          const Item I = load_item(a, idx, 0);
          // the item's queries are in tensor memory and its first q_rope' is written
          ok = wait_bar<true>(c, B_QREADY, item & 1) && wait_bar<true>(c, B_ROPE, rope_ev++ & 1);
          int prev_seg = -1;
          KeyTile cur{0, 0, 0, -1};
          bool have = next_tile(cur, I);
          while (ok && have) {
            const int b = j & 1;
            ok = wait_bar<true>(c, B_SFREE + b, ((j >> 1) & 1) ^ 1);
            if (ok && prev_seg >= 0 && cur.j != prev_seg)
              ok = wait_bar<true>(c, B_ROPE, rope_ev++ & 1);
            if (!ok) break;
            tc::tc_fence_after();
            const uint32_t ts = tbase + T_S + 128 * b;
            const int slot = cnt % KRING;
            ok = wait_bar(c, B_KFULL + slot, (cnt / KRING) & 1);
            if (!ok) break;
            tc::tc_fence_after();
            const uint32_t base = ka + slot * KSLOT;
            KeyTile nx = cur;
            const bool have_next = next_tile(nx, I);
            // B = K[64 keys of each CTA x 16 dims]: the rope chunk first (q_rope'
            // hi and lo), then the nope chunks
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t bd = tc::sdesc_sw128(base + NCH * HCHUNK + 32 * k, 16, 1024);
              tc::mma_ss_2sm(ts, tc::sdesc_sw128(ropa + 32 * k, 16, 1024), bd, idS, k != 0);
              tc::mma_ss_2sm(ts, tc::sdesc_sw128(ropa + CHUNK + 32 * k, 16, 1024), bd, idS, 1);
            }
            // the last tile of a segment or of the item: the rope warps may
            // rewrite q_rope' for the next segment (or item) once these rope
            // MMAs are done, while the nope MMAs below still run
            if (!have_next || nx.j != cur.j) tc::mma_commit_2sm(&bar[B_SWITCH], 0x3);
#pragma unroll
            for (int cc = 0; cc < NCH; ++cc)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                tc::mma_ts_2sm(ts, tbase + T_Q + 8 * (4 * cc + k),
                               tc::sdesc_sw128(base + cc * HCHUNK + 32 * k, 16, 1024), idS, 1);
            tc::mma_commit_2sm(&bar[B_KEMPTY + slot], 0x3);
            ++cnt;
            tc::mma_commit_2sm(&bar[B_SFULL + b], 0x3);
            prev_seg = cur.j;
            ++j;
            cur = nx;
            have = have_next;
          }
        }
        tc::mma_commit_2sm(&bar[B_SFINAL], 0x3);
      }
    } else if (warp >= 6) {
      // ------------------------------------- S pair: rope writers -------
      // q_rope' = R(-delta) q_rope as bf16 hi and lo rows of two K-major
      // 128-byte-swizzled operands (RedKnot-MLA paper, RoPE-orthogonality
      // paragraph), rewritten at every segment switch of the key walk as
      // soon as the rope MMAs of the old segment's last tile are done (each
      // tile's chain takes the rope chunk first, so the rewrite overlaps that
      // tile's nope MMAs); each lane keeps the raw q_rope of its two rows in
      // registers
      const int m0 = 64 * (warp - 6) + lane;
      uint32_t sw_ev = 0;
      for (int item = 0;; ++item) {
        const int idx = tt::claimed<4, 0>(c, a.wq, item, a.num_tc_pairs);
        if (idx < 0) break;
        const Item I = load_item(a, idx, r);
        uint32_t raw[2][32];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const tt::RowInfo ri = tt::row_info(a, I.t, I.rq, m0 + 32 * e);
          const uint16_t* qrow = ri.p >= 0 ? a.q + (ri.frow * a.H + ri.head) * DK : nullptr;
          if (qrow) {
            const uint4* s4 = reinterpret_cast<const uint4*>(qrow + 64 * NCH);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint4 v = __ldg(s4 + u);
              raw[e][4 * u] = v.x;
              raw[e][4 * u + 1] = v.y;
              raw[e][4 * u + 2] = v.z;
              raw[e][4 * u + 3] = v.w;
            }
          } else {
#pragma unroll
            for (int u = 0; u < 32; ++u) raw[e][u] = 0;
          }
        }
        auto put_rope = [&](int seg) {
          const float4* cs4 =
              reinterpret_cast<const float4*>(a.rope_cs + static_cast<int64_t>(I.rq.seg_first + seg) * 64);
          // one row per pass (not unrolled: the body is long)
#pragma unroll 1
          for (int e = 0; e < 2; ++e) {
            const int m = m0 + 32 * e;
            const uint32_t sw = static_cast<uint32_t>(m & 7);
            uint8_t* rrow = sm + OFF_ROPE + m * 128;
            uint32_t cur[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) cur[i] = e ? raw[1][i] : raw[0][i];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              uint32_t hi[4], lo[4];
#pragma unroll
              for (int v2 = 0; v2 < 2; ++v2) {
                const float4 w = __ldg(cs4 + 2 * u + v2);  // (cos, sin) of pairs 4u + 2 v2, + 1
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int jj = 4 * u + 2 * v2 + h;
                  const float co = h ? w.z : w.x, si = h ? w.w : w.y;
                  const float x = __uint_as_float(cur[jj] << 16);
                  const float y = __uint_as_float(cur[jj] & 0xffff0000u);
                  const float xr = fmaf(x, co, y * si), yr = fmaf(-x, si, y * co);
                  const uint32_t hw = pack_bf16x2(xr, yr);
                  hi[2 * v2 + h] = hw;
                  lo[2 * v2 + h] = pack_bf16x2(xr - __uint_as_float(hw << 16),
                                               yr - __uint_as_float(hw & 0xffff0000u));
                }
              }
              *reinterpret_cast<uint4*>(rrow + ((u ^ sw) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
              *reinterpret_cast<uint4*>(rrow + CHUNK + ((u ^ sw) << 4)) =
                  make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
          }
          tc::fence_proxy_async();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive_cluster(cbar(B_ROPE, 0));
        };
        KeyTile kt{0, 0, 0, -1};
        bool have = next_tile(kt, I);
        // a later item: the previous item's last rope MMAs are done first
        if (item > 0) {
          if (!__all_sync(0xffffffffu, wait_bar(c, B_SWITCH, sw_ev++ & 1))) break;
          tc::tc_fence_after();
        }
        int seg = have ? kt.j : -1;  // the segment to write q_rope' for next
        bool ok = true;
        while (seg >= 0) {
          put_rope(seg);  // one call site: the body is large
          seg = -1;
          while (have) {
            KeyTile nx = kt;
            const bool have_next = next_tile(nx, I);
            const bool sw = have_next && nx.j != kt.j;
            kt = nx;
            have = have_next;
            if (sw) {
              // the old segment's rope MMAs are done: none reads q_rope' any more
              if (__all_sync(0xffffffffu, wait_bar(c, B_SWITCH, sw_ev++ & 1))) {
                tc::tc_fence_after();
                seg = kt.j;
              } else {
                have = false;
                ok = false;
              }
              break;
            }
          }
        }
        if (!ok) break;
      }
    } else {
      // ------------------- S pair: queries, rotation and online softmax ---
      const int quarter = warp & 3;
      const int m = quarter * 32 + lane;
      const bool issuer = tid == 64;  // issues the bulk copies of P
      const uint32_t lt = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
      const float sl2 = a.scale_log2;
      const int sink = a.sink, window = a.window;
      const uint32_t orank = crank + 2;
      const uint32_t sw = static_cast<uint32_t>(m & 7);
      int j = 0;  // tiles of the walk so far, over all items
      bool ok = true;
      for (int item = 0; ok; ++item) {
        const int idx = tt::claimed<4, 0>(c, a.wq, item, a.num_tc_pairs);
        if (idx < 0) break;
        const Item I = load_item(a, idx, r);
        const tt::RowInfo ri = tt::row_info(a, I.t, I.rq, m);
        const uint16_t* qrow = ri.p >= 0 ? a.q + (ri.frow * a.H + ri.head) * DK : nullptr;
        // this lane's nope queries -> tensor memory (32-bit column c = dims 2c,
        // 2c + 1).  The loads are coalesced: in step u a warp reads four whole
        // 128-byte rows of a chunk (lane l: 16-byte unit l & 7 of row 4u + l / 8
        // of the warp's 32 rows), and a 4 KB slice of the P staging buffer
        // (unused until the first P) turns them back into one row per lane;
        // four chunks' loads in flight at a time.  The last S of the previous
        // item has been read, so its MMAs no longer read the queries; in a
        // later item the slices are written only once every P half sent so far
        // has landed (the copies read the staging slots)
        {
          bool okq = true;
          uint8_t* qs = sm + OFF_STG + quarter * 4096;
          const int rsub = lane >> 3, unit = lane & 7;
          const uint4* qsrc[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            qsrc[u] = reinterpret_cast<const uint4*>(__shfl_sync(
                0xffffffffu, reinterpret_cast<unsigned long long>(qrow), 4 * u + rsub));
#pragma unroll 1
          for (int i0 = 0; i0 < NCH; i0 += 4) {
            uint4 qw[4][8];
#pragma unroll
            for (int ii = 0; ii < 4; ++ii)
#pragma unroll
              for (int u = 0; u < 8; ++u)
                qw[ii][u] = (qsrc[u] && i0 + ii < NCH) ? __ldg(qsrc[u] + 8 * (i0 + ii) + unit)
                                                       : make_uint4(0u, 0u, 0u, 0u);
            if (i0 == 0 && item > 0) {
              if (lane == 0) okq = wait_count(c, &misc[2], static_cast<uint32_t>(2 * j));
              okq = __shfl_sync(0xffffffffu, okq ? 1 : 0, 0) != 0;
            }
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
              if (i0 + ii >= NCH) break;
              if (okq) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  const int row = 4 * u + rsub;
                  *reinterpret_cast<uint4*>(qs + row * 128 + ((unit ^ (row & 7)) << 4)) = qw[ii][u];
                }
              }
              __syncwarp();
              uint32_t v[32];
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint4 x = *reinterpret_cast<const uint4*>(qs + lane * 128 + ((k ^ (lane & 7)) << 4));
                v[4 * k] = x.x;
                v[4 * k + 1] = x.y;
                v[4 * k + 2] = x.z;
                v[4 * k + 3] = x.w;
              }
              __syncwarp();
              tc::tmem_st32(lt + T_Q + 32 * (i0 + ii), v);
            }
          }
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_cluster(cbar(B_QREADY, 0));
        KeyTile kt{0, 0, 0, -1};
        bool have = next_tile(kt, I);
        float m_run = -INFINITY, l_run = 0.f;
        // Every wait below is bounded; a failed wait skips the work but the
        // lane still reaches the per-tile vote, so the four warps leave the
        // loop together and no lane is left at a named barrier.
        while (ok && have) {
          const int b = j & 1;
          KeyTile nx = kt;
          // the next key tile: found while this tile's loads of S are in
          // flight (the rotary-value kernel, measured slower that way, finds
          // it first)
          bool have_next = VROPE ? next_tile(nx, I) : false;
          bool okw = __all_sync(0xffffffffu, wait_bar(c, B_SFULL + b, (j >> 1) & 1));
          uint32_t s[4][32];
          float alpha = 1.f;
          if (okw) {
            tc::tc_fence_after();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tc::tmem_ld32(lt + T_S + 128 * b + 32 * q4, s[q4]);
            if (!VROPE) have_next = next_tile(nx, I);
            tc::tmem_wait_ld();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_cluster(cbar(B_SFREE + b, 0));
            // the landed-halves count, read before the softmax: the halves of
            // tile j - 1 have usually landed by then, and the wait below then
            // needs only its acquire fence (the rotary-value kernel, at its
            // register limit, polls after the softmax only)
            const uint32_t landed = (!VROPE && issuer) ? tc::ld_relaxed_cluster_u32(&misc[2]) : 0u;

            // scores are scaled inside the exponent: x = s * scale * log2(e)
            alpha = tt::softmax_tile(s, kt, ri, sink, window, sl2, m_run, l_run);
            // the O pair's P buffer b is free once the output MMAs of tile
            // j - 2 are done
            okw = __all_sync(0xffffffffu, wait_bar(c, B_PEMPTY + b, ((j >> 1) & 1) ^ 1));
            // P half k = 2j + h of the walk is staged in slot k % 3, whose last
            // copy (half k - 3) must have landed: a shared::cta ->
            // shared::cluster bulk copy completes on the receiver's barrier
            // only, so the output CTA counts the halves that have landed
            if (okw && issuer && j > 0) {
              if (!VROPE && landed >= static_cast<uint32_t>(2 * j - 1))
                tc::fence_acquire_cluster_smem();
              else
                okw = wait_count(c, &misc[2], static_cast<uint32_t>(2 * j - 1));
            }
          }
          ok = tc::named_and(1, 128, okw);
          if (!ok) break;
          const int k0 = (2 * j) % NSTG;
          uint8_t* stg[2] = {sm + OFF_STG + k0 * CHUNK, sm + OFF_STG + (k0 == NSTG - 1 ? 0 : k0 + 1) * CHUNK};
          // lane m's 128 keys: two 64-key halves of 8 16-byte units, 128-byte swizzle
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4*>(stg[h] + m * 128 + ((u ^ sw) << 4)) =
                  make_uint4(s[h][4 * u], s[h][4 * u + 1], s[h][4 * u + 2], s[h][4 * u + 3]);
          // the lane's record goes straight to the output CTA, counted with the second half
          const uint32_t pdst = tc::mapa_shared(smem_u32(sm + OFF_P + b * PSTRIDE), orank);
          tc::st_async_v2f32(pdst + PBUF + m * 8, alpha, l_run, cbar(B_PFULL1 + b, orank));
          tc::fence_proxy_async();
          tc::named_sync(1, 128);
          if (issuer) {
            tc::bulk_copy_to_cluster(pdst, smem_u32(stg[0]), CHUNK, cbar(B_PFULL0 + b, orank));
            tc::bulk_copy_to_cluster(pdst + CHUNK, smem_u32(stg[1]), CHUNK, cbar(B_PFULL1 + b, orank));
          }
          ++j;
          kt = nx;
          have = have_next;
        }
        if (ok && ri.store && l_run > 0.f)
          a.lse[ri.frow * a.H + ri.head] = tt::lse_of(m_run, l_run);
      }
      // every output MMA has consumed its P before the cluster may exit
      for (int jj = j - 1; ok && jj >= 0 && jj >= j - 2; --jj)
        ok = __all_sync(0xffffffffu, wait_bar(c, B_PEMPTY + (jj & 1), (jj >> 1) & 1));
    }
  } else {
    if (warp == 0) {
      // ------------------------------------------- O pair: TMA producer --
      if (lane == 0) {
        uint32_t cnt = 0;
        bool ok = true;
        for (int item = 0; ok; ++item) {
          const int idx = tt::claimed<4, 0>(c, a.wq, item, a.num_tc_pairs);
          if (idx < 0) break;
          const Item I = load_item(a, idx, r);
          KeyTile cur{0, 0, 0, -1};
          bool have = next_tile(cur, I);
          while (ok && have) {
            const int slot = cnt % VRING;
            ok = wait_bar(c, B_VEMPTY + slot, ((cnt / VRING) & 1) ^ 1);
            if (!ok) break;
            if (r == 0) tc::mbar_arrive_expect_tx(&bar[B_VFULL + slot], 2 * VSLOT);
            // value columns 256 r .. 256 r + 255 (chunks 4 r .. 4 r + 3)
            tc::tma_load_3d_2sm(smem_u32(sm + OFF_VRING + slot * VSLOT),
                                a.segmaps + kSegMaps * (I.rq.seg_first + cur.j) + MAP_V4,
                                cbar(B_VFULL + slot, 2), 0, cur.k0 - I.segs[cur.j].delta,
                                4 * static_cast<int>(r));
            ++cnt;
            have = next_tile(cur, I);
          }
        }
        if (r == 0)
          for (uint32_t k = (cnt > VRING ? cnt - VRING : 0); k < cnt; ++k)
            drain_bar(c, B_VFULL + k % VRING, (k / VRING) & 1);
      }
    } else if (warp == 1) {
      // ------------------------------ O pair: MMA issuer (rank 2 only) --
      if (lane == 0 && r == 0) {
        const uint32_t idPV = tc::idesc_bf16(256, 256, false, true);
        const uint32_t pa = smem_u32(sm + OFF_P), va = smem_u32(sm + OFF_VRING);
        uint32_t cnt = 0;
        int j = 0;
        bool ok = true;
        for (int item = 0; ok; ++item) {
          const int idx = tt::claimed<4, 0>(c, a.wq, item, a.num_tc_pairs);
          if (idx < 0) break;
          const Item I = load_item(a, idx, 0);
          KeyTile cur{0, 0, 0, -1};
          bool have = next_tile(cur, I);
          // the item's first output MMA starts the accumulator afresh; its
          // P-ready wait comes after the lanes' epilogue reads of the previous
          // item (program order on their side)
          bool first = true;
          while (ok && have) {
            const int b = j & 1;
            ok = wait_bar<true>(c, B_PREADY + b, (j >> 1) & 1);
            if (!ok) break;
            tc::tc_fence_after();
            const int slot = cnt % VRING;
            ok = wait_bar(c, B_VFULL + slot, (cnt / VRING) & 1);
            if (!ok) break;
            tc::tc_fence_after();
            const uint32_t base = va + slot * VSLOT;
            // A = P[128 lanes of each CTA x 16 keys]; B = V[16 keys x 256
            // columns]: 128 from each CTA, two 64-column chunks 16 KB apart.
            // Output columns 256 v + 128 h + i hold value column
            // 256 h + 128 v + i (h: the CTA that supplied them).
#pragma unroll
            for (int v = 0; v < 2; ++v)
#pragma unroll
              for (int k = 0; k < 8; ++k)
                tc::mma_ss_2sm(tbase + T_O + 256 * v,
                               tc::sdesc_sw128(pa + b * PSTRIDE + (k >> 2) * CHUNK + 32 * (k & 3), 16, 1024),
                               tc::sdesc_sw128(base + 2 * CHUNK * v + 2048 * k, CHUNK, 1024), idPV,
                               (!first || k > 0) ? 1u : 0u);
            tc::mma_commit_2sm(&bar[B_VEMPTY + slot], 0xC);
            ++cnt;
            tc::mma_commit_2sm(&bar[B_ODONE], 0xC);
            tc::mma_commit_2sm(&bar[B_PEMPTY + b], 0x3);
            ++j;
            first = false;
            have = next_tile(cur, I);
          }
          if (ok) tc::mma_commit_2sm(&bar[B_OFINAL], 0xC);  // one phase per item
        }
        tc::mma_commit_2sm(&bar[B_SFINAL], 0xC);  // the pipe is empty before teardown
      }
    } else if (warp == 6) {
      // ------------- O pair: counts the sender's P halves that have landed
      // (a thread of its own, so that the count never waits for the rescale
      // / turn work of the lanes), with a release store into the sender's
      // counter.  It cannot fall two phases behind on a P barrier: tile
      // j + 2 is sent only after the count has passed tile j + 1's first half.
      if (lane == 0) {
        int j = 0;
        const uint32_t cnt = tc::mapa_shared(smem_u32(&misc[2]), crank - 2);
        bool ok = true;
        for (int item = 0; ok; ++item) {
          const int idx = tt::claimed<4, 0>(c, a.wq, item, a.num_tc_pairs);
          if (idx < 0) break;
          const Item I = load_item(a, idx, r);
          KeyTile kt{0, 0, 0, -1};
          bool have = next_tile(kt, I);
          while (have) {
            const uint32_t par = (j >> 1) & 1;
            ok = wait_bar<true>(c, B_PFULL0 + (j & 1), par);
            if (!ok) break;
            tc::st_release_cluster_u32(cnt, static_cast<uint32_t>(2 * j + 1));
            ok = wait_bar<true>(c, B_PFULL1 + (j & 1), par);
            if (!ok) break;
            tc::st_release_cluster_u32(cnt, static_cast<uint32_t>(2 * j + 2));
            ++j;
            have = next_tile(kt, I);
          }
        }
      }
    } else if (warp < 6) {
      // ------------------------------- O pair: rescale and epilogue ------
      const int quarter = warp & 3;
      const int m = quarter * 32 + lane;
      const uint32_t lt = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
      int j = 0;  // tiles of the walk so far, over all items
      bool ok = true;
      for (int item = 0; ok; ++item) {
        const int idx = tt::claimed<4, 0>(c, a.wq, item, a.num_tc_pairs);
        if (idx < 0) break;
        const Item I = load_item(a, idx, r);
        const tt::RowInfo ri = tt::row_info(a, I.t, I.rq, m);
        float l_fin = 0.f;
        KeyTile kt{0, 0, 0, -1};
        bool have = next_tile(kt, I);
        // rotary value: the segment whose canonical frame the output's rope
        // columns (448..511, output column = value column there) are in
        int seg_frame = kt.j;
        while (ok && have) {
          const int b = j & 1;
          ok = __all_sync(0xffffffffu, wait_bar<true>(c, B_PFULL0 + b, (j >> 1) & 1) &&
                                           wait_bar<true>(c, B_PFULL1 + b, (j >> 1) & 1));
          if (!ok) break;
          const volatile float* rp =
              reinterpret_cast<const volatile float*>(sm + OFF_P + b * PSTRIDE + PBUF + m * 8);
          const float alpha = rp[0];
          l_fin = rp[1];
          // arm buffer b for tile j + 2 (its copy starts after the MMAs of tile j)
          if (m == 0) {
            tc::mbar_arrive_expect_tx(&bar[B_PFULL0 + b], CHUNK);
            tc::mbar_arrive_expect_tx(&bar[B_PFULL1 + b], CHUNK + RBUF);
          }
          const bool scale = __any_sync(0xffffffffu, alpha != 1.f);
          const bool turn = VROPE && kt.j != seg_frame;
          if (scale || turn) {
            // the output MMAs of tile j - 1 finish before O is rescaled / turned
            if (j >= 1) ok = __all_sync(0xffffffffu, wait_bar(c, B_ODONE, (j - 1) & 1));
            if (!ok) break;
            tc::tc_fence_after();
            // a new segment: R(delta_frame - delta_next) moves the rope columns
            // into the next segment's canonical frame
            const float4* ca = reinterpret_cast<const float4*>(a.rope_cs + int64_t(I.rq.seg_first + seg_frame) * 64);
            const float4* cb = reinterpret_cast<const float4*>(a.rope_cs + int64_t(I.rq.seg_first + kt.j) * 64);
#pragma unroll 1
            for (int q8 = scale ? 0 : 14; q8 < 16; ++q8) {
              uint32_t o[32];
              tc::tmem_ld32(lt + T_O + 32 * q8, o);
              tc::tmem_wait_ld();
              if (scale) {
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              }
              if (turn && q8 >= 14) tt::turn16(o, ca, cb, 16 * (q8 - 14));
              tc::tmem_st32(lt + T_O + 32 * q8, o);
            }
            tc::tmem_wait_st();
          }
          seg_frame = kt.j;
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive_cluster(cbar(B_PREADY + b, 2));
          ++j;
          have = next_tile(kt, I);
        }
        if (ok) ok = __all_sync(0xffffffffu, wait_bar(c, B_OFINAL, item & 1));
        tc::tc_fence_after();
        if (ok) {
          const bool st = ri.store && l_fin > 0.f;
          const float inv = st ? 1.f / l_fin : 0.f;
          uint16_t* dst = st ? a.out + (ri.frow * a.H + ri.head) * 512 : nullptr;
          // two 32-column loads per wait; the rows go straight to global memory
          // (the value ring and P buffers already serve the next item)
#pragma unroll 1
          for (int q0 = 0; q0 < 16; q0 += 2) {
            uint32_t o[2][32];
            tc::tmem_ld32(lt + T_O + 32 * q0, o[0]);
            tc::tmem_ld32(lt + T_O + 32 * (q0 + 1), o[1]);
            tc::tmem_wait_ld();
            if (VROPE && st && q0 == 14) {
              // rotary value: R(delta_frame - p) restores the last segment's
              // output phase and applies the inverse output RoPE at the row's
              // position p (cos / sin of p theta from the two-level table)
              const float4* ca = reinterpret_cast<const float4*>(a.rope_cs + int64_t(I.rq.seg_first + seg_frame) * 64);
              const float4* ph = reinterpret_cast<const float4*>(a.pos_cs_hi + int64_t(ri.p >> 8) * 64);
              const float4* pl = reinterpret_cast<const float4*>(a.pos_cs_lo + int64_t(ri.p & 255) * 64);
              tt::restore16(o[0], ca, ph, pl, 0);
              tt::restore16(o[1], ca, ph, pl, 16);
            }
            if (st) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int c0 = 32 * (q0 + h);
                const int col = 256 * ((c0 >> 7) & 1) + 128 * (c0 >> 8) + (c0 & 127);
                uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  uint4 w;
                  w.x = pack_bf16x2(__uint_as_float(o[h][8 * u + 0]) * inv, __uint_as_float(o[h][8 * u + 1]) * inv);
                  w.y = pack_bf16x2(__uint_as_float(o[h][8 * u + 2]) * inv, __uint_as_float(o[h][8 * u + 3]) * inv);
                  w.z = pack_bf16x2(__uint_as_float(o[h][8 * u + 4]) * inv, __uint_as_float(o[h][8 * u + 5]) * inv);
                  w.w = pack_bf16x2(__uint_as_float(o[h][8 * u + 6]) * inv, __uint_as_float(o[h][8 * u + 7]) * inv);
                  d4[u] = w;
                }
              }
            }
          }
        }
        // rank 2 reports the items it has finished: the claimer reuses a ring
        // entry only once these are 16 items past its last reader
        if (r == 0 && m == 0)
          tc::st_release_cluster_u32(tc::mapa_shared(smem_u32(&misc[3]), 0),
                                     static_cast<uint32_t>(item + 1));
      }
    }
  }

  // ------------------------------------------------------------ teardown --
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) drain_bar(c, B_SFINAL, 0);  // the pair's MMA pipe is empty
  __syncthreads();
  tc::cluster_sync();  // no CTA leaves while another may still use its memory
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc_2sm(tbase, 512);
  }
}

// Clusters of one launch: as many as the device holds at once (asked once
// per device), never more than there are tile pairs or queue rings.
template <int NCH, bool VROPE>
cudaError_t clusters_t(const KernelArgs& a, int64_t& clusters) {
  auto k = dense_tc4_kernel<NCH, VROPE>;
  clusters = 0;
  static int resident[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int ncl = (dev >= 0 && dev < 64) ? resident[dev] : 0;
  if (ncl <= 0) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4 * 64);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    e = cudaOccupancyMaxActiveClusters(&ncl, k, &cfg);
    if (e != cudaSuccess) return e;
    if (ncl <= 0) return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < 64) resident[dev] = ncl;
  }
  clusters = std::min<int64_t>(std::min<int64_t>(ncl, kQueueClusters), a.num_tc_pairs);
  return cudaSuccess;
}

template <int NCH, bool VROPE>
cudaError_t launch_tc4_t(const KernelArgs& a, cudaStream_t s) {
  auto k = dense_tc4_kernel<NCH, VROPE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  // persistent clusters that claim pairs from the launch's work queue (a.wq,
  // zeroed before the launch)
  int64_t clusters = 0;
  e = clusters_t<NCH, VROPE>(a, clusters);
  if (e != cudaSuccess) return e;
  if (!a.wq) return cudaErrorInvalidValue;  // the work queue lives in the workspace
  if (clusters <= 0) return cudaSuccess;
  k<<<static_cast<unsigned>(4 * clusters), THREADS, SMEM_BYTES, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dense_tc4(const rk_seg_attn_plan_s& p, const KernelArgs& a, const void* q,
                             cudaStream_t s) {
  (void)q;
  if (p.v_rope) return launch_tc4_t<7, true>(a, s);
  return launch_tc4_t<8, false>(a, s);
}

cudaError_t dense_tc4_clusters(const rk_seg_attn_plan_s& p, const KernelArgs& a,
                               int64_t& clusters) {
  if (p.v_rope) return clusters_t<7, true>(a, clusters);
  return clusters_t<8, false>(a, clusters);
}

}  // namespace rk
