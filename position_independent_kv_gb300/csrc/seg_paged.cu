// SegPagedAttention for grouped-query attention on the tcgen05 path.
//
// RedKnot blog ("RedKnot, explained"), "Insight 3: savings must show up in
// memory": the KV cache is stored per KV head in pages; a Global head keeps
// the pages of the whole prompt, a Local head only those of its sink and
// window, so attention needs no mask over the prompt.  Visibility follows
// "Insight 1": Global heads see every k <= p, Local heads k <= p with
// k < sink or k >= p - w.
//
// A sub-tile is 128 query pairs: 128 / G consecutive rows x the G query heads
// of one KV head, so every key page is read once for the whole group.  Three
// kernels share the tile list format:
//
// seg_paged_two_kernel, for tiles with more than 64 pairs in use (never
// split): a tile is two sub-tiles (the second the next 128 / G rows) that walk the union of
// their key blocks, so a page serves 2 x 128 / G rows.  One CTA per tile
// (320 threads):
//   warp 0     TMA producer: for each key block its K page, then its V page
//              (each a 32 KB box of 128 tokens x 128 dims, chunk-major,
//              128-byte swizzled), through a four-slot ring.
//   warp 1     MMA issuer, alternating the sub-tiles A and B so that one's
//              softmax runs under the other's MMAs: PV_A(j), S_A(j+1),
//              PV_B(j), S_B(j+1), ... with S_X = Q_X K^T (M = 128, N = 128
//              keys, A = Q_X and B = K from shared memory) and O_X += P_X V
//              (A = P_X from tensor memory, B = V in MN-major form).
//   warps 2-5  sub-tile A, warps 6-9 sub-tile B: one thread per query pair
//              (its TMEM lane) writes its query row into shared memory, masks
//              the edge blocks, keeps the running max in the log2 domain with
//              a lazy rescale of O when it grows by more than 2^8, writes P
//              (bf16) over the first half of its S columns, and finally
//              normalises and stores O and the LSE.
// Tensor memory (512 columns): S_A / P_A (128) | S_B / P_B (128) | O_A (128) |
// O_B (128).  P_X overwrites S_X after the lanes have read it; the next S_X
// is issued after the P.V that reads P_X, and the MMAs of one thread run in
// issue order.
//
// seg_paged_one_kernel, for tiles with 17 to 64 pairs in use (the last rows
// of a request): one sub-tile per CTA whose query pairs each have two lane threads,
// one per warpgroup, taking half of a block's keys and half of the output
// columns (the row max is agreed through shared memory with a per-block
// bar.red vote that also lets every warp leave together after a failed
// wait); Q in tensor memory, S double-buffered, a six-slot K/V ring.  A long
// walk is split into parts of 32 blocks on separate CTAs; each part leaves
// its normalised partial output and LSE in the workspace and the last part
// merges them by log-sum-exp (parts without a visible key weigh 0).
//
// seg_paged_dec_kernel, for tiles with at most 16 pairs in use (decode
// steps): a persistent mma.sync kernel, one CTA per SM, with the pairs on
// the 16-row side of the tile and each of eight warps owning 16 keys of
// every block (details at the kernel); walks of more than 48 blocks are
// split into parts of 32 blocks, merged like the one-sub-tile kernel's.
// Every wait is bounded (2 s); on expiry the CTA records
// RK_ERR_DEVICE_TIMEOUT and every role stops; the producer waits (bounded)
// for its copies in flight and tensor memory is released after the MMA pipe
// has drained.

#include <algorithm>
#include <climits>
#include <cmath>
#include <map>
#include <new>
#include <vector>

#include "rk_seg_paged.h"
#include "tc_tile.cuh"

namespace rk {
namespace sp {

constexpr int PAGE = 128;                   // tokens per page (= keys per block)
constexpr int DH = 128;                     // head dim
constexpr uint32_t CHUNK = 16384;           // 128 rows x 64 bf16

struct Req {
  int32_t T;
  int32_t q_row_begin;
  int64_t row_base;      // first flattened row of the request
  int64_t table_off;     // offset of the request's [Hkv][max_blocks] block table
  int64_t blk_off;       // offset of the request's [max_blocks] offset indices
};

// rows (up to 2 x 128 / G) from p0 of KV head g: sub-tile A the first
// 128 / G of them, sub-tile B the rest; the key walk is blocks
// [0, sink_blocks) then [win_lo, hi] (sink_blocks = 0: [win_lo, hi] only),
// and this CTA takes walk steps [jb, je).  A split tile's parts are
// part_first .. part_first + nparts - 1; their partials sit at workspace
// lanes lane0 + (part - part_first) * rows * G + m.
struct Tile {
  int32_t req, g, p0, rows;
  int32_t sink_blocks, win_lo, hi, jb;
  int32_t je, part, part_first, nparts;
  int32_t group, lane0, pad0, pad1;
};

struct Args {
  const uint16_t* q;
  const Tile* tiles;
  const Req* reqs;
  const int32_t* table;
  const uint8_t* role;
  uint16_t* out;
  float* lse;
  int32_t* status;
  int32_t Hq, G, max_blocks;
  int32_t sink, window;
  float scale_log2;
  int32_t num_tiles;     // tiles of the launch (the decode kernel strides over them)
  float* ws_o;           // [lanes][128] normalised partial outputs of split tiles
  float* ws_lse;         // [lanes]
  int32_t* ws_ticket;    // [split tiles]
  const int32_t* blk_cs; // relocated documents: [R][max_blocks] index of the block's offset
                         // (index 0 is the zero offset)
  const float* cs;       // [offsets][64][2] cos, sin of delta * theta_j
};

struct Maps {
  CUtensorMap k, v;
};

__device__ __forceinline__ int block_of(const Tile& t, int j) {
  return j < t.sink_blocks ? j : t.win_lo + (j - t.sink_blocks);
}

// Log-sum-exp merge of a split tile's parts (RedKnot-MLA paper, the
// numerically stable merge of the RoPE-orthogonality paragraph): every part
// left its normalised output and its natural-log LSE at workspace lanes
// lane0 + part * nl + pair; parts without a visible key (LSE -inf) weigh 0.
// Run by the last part to finish, spread over `nthr` threads (item = pair,
// group of 8 dims).
__device__ void merge_parts(const Args& a, const Tile& t, const Req& rq, int tid, int nthr) {
  const int nl = t.rows * a.G;
  for (int it = tid; it < nl * 16; it += nthr) {
    const int l = it >> 4, d0 = (it & 15) * 8;
    const int64_t s0 = int64_t(t.lane0) + l;
    float mxp = -INFINITY;
    for (int q = 0; q < t.nparts; ++q) mxp = fmaxf(mxp, __ldcg(a.ws_lse + s0 + int64_t(q) * nl));
    float wsum = 0.f;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int q = 0; q < t.nparts; ++q) {
      const float lq = __ldcg(a.ws_lse + s0 + int64_t(q) * nl);
      if (lq == -INFINITY) continue;
      const float wq = __expf(lq - mxp);
      wsum += wq;
      const float4* src = reinterpret_cast<const float4*>(a.ws_o + (s0 + int64_t(q) * nl) * DH + d0);
      const float4 x = __ldcg(src), y = __ldcg(src + 1);
      acc[0] += wq * x.x; acc[1] += wq * x.y; acc[2] += wq * x.z; acc[3] += wq * x.w;
      acc[4] += wq * y.x; acc[5] += wq * y.y; acc[6] += wq * y.z; acc[7] += wq * y.w;
    }
    const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int lr = l / a.G, lh = l - lr * a.G;
    const int64_t orow = rq.row_base + (t.p0 + lr - rq.q_row_begin);
    const int ohead = t.g * a.G + lh;
    uint4 v;
    v.x = pack_bf16x2(acc[0] * winv, acc[1] * winv);
    v.y = pack_bf16x2(acc[2] * winv, acc[3] * winv);
    v.z = pack_bf16x2(acc[4] * winv, acc[5] * winv);
    v.w = pack_bf16x2(acc[6] * winv, acc[7] * winv);
    *reinterpret_cast<uint4*>(a.out + (orow * a.Hq + ohead) * DH + d0) = v;
    if (d0 == 0) a.lse[orow * a.Hq + ohead] = wsum > 0.f ? mxp + logf(wsum) : -INFINITY;
  }
}

// ---- two sub-tiles of 128 pairs per CTA (tiles with more than 64 pairs in use)
namespace two {

constexpr int THREADS = 320;
constexpr int RING = 4;
constexpr uint32_t SLOT = 2 * CHUNK;        // one K or V page
constexpr uint32_t OFF_Q = 0;               // Q_A, Q_B: 2 x 32 KB
constexpr uint32_t OFF_RING = 4 * CHUNK;
constexpr uint32_t OFF_BAR = OFF_RING + RING * SLOT;
enum {
  B_FULL = 0,
  B_EMPTY = RING,
  B_QFULL = 2 * RING,        // queries in shared memory (one arrival per lane warp, 8)
  B_SFULL,                   // 2 (A, B): S_X(j) written
  B_PREADY = B_SFULL + 2,    // 2: P_X(j) written and O_X rescaled (one arrival per warp of X, 4)
  B_ODONE = B_PREADY + 2,    // 2: O_X += P_X(j) V(j) done
  B_FINAL = B_ODONE + 2,
  NBAR
};
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
constexpr uint32_t T_S = 0, T_O = 256;      // sub-tile X: S/P at 128 X, O at 256 + 128 X

__global__ void __launch_bounds__(THREADS, 1)
    seg_paged_two_kernel(const __grid_constant__ Args a, const __grid_constant__ Maps mp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  const tt::Ctx c{bar, reinterpret_cast<volatile uint32_t*>(misc + 1), a.status};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Tile t = a.tiles[blockIdx.x];
  const Req rq = a.reqs[t.req];
  const int nb = t.je - t.jb;                 // this CTA's walk steps
  const int RT = 128 / a.G;                   // rows of a sub-tile
  const bool has_b = t.rows > RT;             // sub-tile B in use

  if (tid == 0) {
    for (int i = 0; i < RING; ++i) {
      tc::mbar_init(&bar[B_FULL + i], 1);
      tc::mbar_init(&bar[B_EMPTY + i], 1);
    }
    tc::mbar_init(&bar[B_QFULL], 8);
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(&bar[B_SFULL + x], 1);
      tc::mbar_init(&bar[B_PREADY + x], 4);
      tc::mbar_init(&bar[B_ODONE + x], 1);
    }
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
      tc::prefetch_tmap(&mp.k);
      tc::prefetch_tmap(&mp.v);
      const int32_t* tab = a.table + rq.table_off + int64_t(t.g) * a.max_blocks;
      uint32_t cnt = 0;
      bool ok = true;
      auto load = [&](const CUtensorMap* map, int page) {
        const int slot = cnt % RING;
        if (!tt::wait_bar(c, B_EMPTY + slot, ((cnt / RING) & 1) ^ 1)) return false;
        tc::mbar_arrive_expect_tx(&bar[B_FULL + slot], SLOT);
        tc::tma_load_4d(smem_u32(sm + OFF_RING + slot * SLOT), map, &bar[B_FULL + slot], 0, 0, 0,
                        page);
        ++cnt;
        return true;
      };
      // K_j, then V_j: the order in which the issuer first needs them
      for (int j = 0; j < nb && ok; ++j) {
        const int page = tab[block_of(t, t.jb + j)];
        ok = load(&mp.k, page);
        if (ok) ok = load(&mp.v, page);
      }
      // copies in flight land before the CTA may exit
      for (uint32_t k = (cnt > RING ? cnt - RING : 0); k < cnt; ++k)
        tt::drain_bar(c, B_FULL + k % RING, (k / RING) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      bool ok = tt::wait_bar(c, B_QFULL, 0);
      tc::tc_fence_after();
      const uint32_t idS = tc::idesc_bf16(128, 128, false, false);
      const uint32_t idPV = tc::idesc_bf16(128, 128, false, true);
      const uint32_t qa = smem_u32(sm + OFF_Q), ra = smem_u32(sm + OFF_RING);
      const int nx = has_b ? 2 : 1;
      // slot of K_j is 2j mod RING, of V_j 2j + 1 mod RING (loads alternate)
      auto full = [&](uint32_t ld) {
        const bool r = tt::wait_bar(c, B_FULL + ld % RING, (ld / RING) & 1);
        tc::tc_fence_after();
        return r;
      };
      auto score = [&](int x, int j) {
        const uint32_t base = ra + ((2u * j) % RING) * SLOT;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_ss(tbase + T_S + 128 * x,
                       tc::sdesc_sw128(qa + (2 * x + cc) * CHUNK + 32 * k, 16, 1024),
                       tc::sdesc_sw128(base + cc * CHUNK + 32 * k, 16, 1024), idS, (cc | k) != 0);
        tc::mma_commit(&bar[B_SFULL + x]);
      };
      auto pv = [&](int x, int j) {
        const uint32_t base = ra + ((2u * j + 1) % RING) * SLOT;
        // B = V[16 keys x 128 dims]: two 64-dim chunks 16 KB apart (LBO)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tc::mma_ts(tbase + T_O + 128 * x, tbase + T_S + 128 * x + 8 * k,
                     tc::sdesc_sw128(base + 2048 * k, CHUNK, 1024), idPV, (j > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(&bar[B_ODONE + x]);
      };
      if (ok && nb > 0) {
        ok = full(0);
        if (ok) {
          for (int x = 0; x < nx; ++x) score(x, 0);
          tc::mma_commit(&bar[B_EMPTY + 0]);  // K_0 read by every score MMA
        }
      }
      for (int j = 0; j < nb && ok; ++j) {
        ok = full(2u * j + 1);              // V_j
        const bool more = j + 1 < nb;
        for (int x = 0; x < nx && ok; ++x) {
          ok = tt::wait_bar(c, B_PREADY + x, j & 1);
          if (!ok) break;
          tc::tc_fence_after();
          pv(x, j);
          if (more) {
            if (x == 0) ok = full(2u * j + 2);  // K_{j+1}
            if (!ok) break;
            score(x, j + 1);
          }
        }
        if (!ok) break;
        tc::mma_commit(&bar[B_EMPTY + (2u * j + 1) % RING]);          // V_j
        if (more) tc::mma_commit(&bar[B_EMPTY + (2u * j + 2) % RING]);  // K_{j+1}
      }
      tc::mma_commit(&bar[B_FINAL]);
    }
  } else {
    // ------------------------------------------- softmax and epilogue ----
    const int lw = warp - 2;           // 0..7
    const int x = lw >> 2;             // sub-tile
    const int quarter = warp & 3;      // TMEM lane quarter this warp may access
    const int m = quarter * 32 + lane;
    const int r = m / a.G, h = m - r * a.G;
    const int p = t.p0 + x * RT + r;
    const bool active = x == 0 || has_b;  // this warpgroup's sub-tile exists
    const bool valid = x * RT + r < t.rows;
    const bool glob = a.role[t.g] != 0;
    const uint32_t lt = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t tS = lt + T_S + 128 * x, tO = lt + T_O + 128 * x;
    const float sl2 = a.scale_log2;
    const int sink = a.sink, window = a.window;
    const int64_t row = rq.row_base + (p - rq.q_row_begin);
    const int head = t.g * a.G + h;
    // this lane's query row -> shared memory: two 64-dim chunks of 128 rows,
    // 128-byte swizzle (A operand of the score MMAs); rows past the tile's
    // end are zero
    {
      const uint4* src = valid ? reinterpret_cast<const uint4*>(a.q + (row * a.Hq + head) * DH)
                               : nullptr;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint4 v = src ? __ldg(src + u) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sm + OFF_Q + (2 * x + (u >> 3)) * CHUNK + m * 128 +
                                  (((u & 7) ^ (m & 7)) << 4)) = v;
      }
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[B_QFULL]);
    }
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = active;
    for (int j = 0; j < nb && ok; ++j) {
      const int k0 = block_of(t, t.jb + j) * PAGE;
      ok = __all_sync(0xffffffffu, tt::wait_bar(c, B_SFULL + x, j & 1));
      if (!ok) break;
      tc::tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tc::tmem_ld32(tS + 32 * q4, s[q4]);
      tc::tmem_wait_ld();
      // every key of the block visible for this row?  (then no masks)
      const bool full = valid && k0 + PAGE - 1 <= p &&
                        (glob || k0 >= p - window || k0 + PAGE <= sink);
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
            const int key = k0 + 32 * q4 + i;
            bool vis = valid && key <= p;
            if (!glob) vis = vis && (key < sink || key >= p - window);
            const float xv = vis ? __uint_as_float(s[q4][i]) : -INFINITY;
            s[q4][i] = __float_as_uint(xv);
            mx4[i & 3] = fmaxf(mx4[i & 3], xv);
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
      const float nbias = (m_run == -INFINITY) ? 0.f : -m_run;
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};
      // P in place: keys 2i, 2i + 1 of column block q4 go to word 16 q4 + i
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(s[q4][2 * i]), sl2, nbias));
          const float p1 = fast_exp2(fmaf(__uint_as_float(s[q4][2 * i + 1]), sl2, nbias));
          ls4[i & 3] += p0 + p1;
          s[q4 >> 1][16 * (q4 & 1) + i] = pack_bf16x2(p0, p1);
        }
      }
      l_run = l_run * alpha + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
      // S_X(j) was issued after P_X(j-1).V, and its completion (above)
      // implies that of every earlier MMA: P and O are free
      tc::tmem_st32(tS, s[0]);
      tc::tmem_st32(tS + 32, s[1]);
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int q8 = 0; q8 < 4; ++q8) {
          uint32_t o[32];
          tc::tmem_ld32(tO + 32 * q8, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tc::tmem_st32(tO + 32 * q8, o);
        }
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[B_PREADY + x]);
    }
    // ---- epilogue ----
    if (ok) ok = __all_sync(0xffffffffu, tt::wait_bar(c, B_FINAL, 0));
    tc::tc_fence_after();
    // tiles of this kernel are never split
    if (ok) {
      const bool st = valid && l_run > 0.f;
      const float inv = st ? 1.f / l_run : 0.f;
      uint16_t* dst = st ? a.out + (row * a.Hq + head) * DH : nullptr;
#pragma unroll 1
      for (int q8 = 0; q8 < 4; ++q8) {
        uint32_t o[32];
        tc::tmem_ld32(tO + 32 * q8, o);
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
      if (st) a.lse[row * a.Hq + head] = m_run * 0.6931471805599453f + logf(l_run);
    }
  }

  // ------------------------------------------------------------ teardown --
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tt::drain_bar(c, B_FINAL, 0);  // the MMA pipe is empty before TMEM is released
    tc::tc_fence_after();
    tc::tmem_dealloc(tbase, 512);
  }
}

}  // namespace two

// ---- one sub-tile, two lane warpgroups (decode steps, split parts, small tiles)
namespace one {

constexpr int THREADS = 320;
constexpr int RING = 6;
constexpr uint32_t SLOT = 2 * CHUNK;        // one K or V page
constexpr uint32_t OFF_RING = 0;
constexpr uint32_t OFF_BAR = OFF_RING + RING * SLOT;
enum {
  B_FULL = 0,
  B_EMPTY = RING,
  B_QFULL = 2 * RING,       // queries in tensor memory (one arrival per lane warp, 8)
  B_SFULL,                   // 2: S buffer j & 1 written
  B_SFREE = B_SFULL + 2,     // 2: S buffer read (one arrival per lane warp, 8)
  B_PREADY = B_SFREE + 2,    // P_j written and O rescaled (one arrival per lane warp, 8)
  B_ODONE,                   // O += P_j V_j done
  B_FINAL,
  NBAR
};
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t OFF_X = (OFF_MISC + 16 + 15) & ~15u;  // row max [2 buffers][2 halves][128], sums [2][128]
constexpr uint32_t SMEM_BYTES = OFF_X + (4 + 2) * 128 * 4 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
constexpr uint32_t T_O = 0, T_S = 128, T_P = 384, T_Q = 448;
// relocated documents: P overwrites the first half of its S buffer (the next
// S into that buffer is issued after the P.V that reads P, and one thread's
// MMAs run in issue order), which frees the columns for the query as bf16
// hi and lo parts of R(-delta) q
constexpr uint32_t T_QH = 384, T_QL = 448;

// Offset index of walk step j of tile t (relocated documents).
__device__ __forceinline__ int32_t cs_of(const Args& a, const Tile& t, const Req& rq, int j) {
  return a.blk_cs[rq.blk_off + block_of(t, t.jb + j)];
}

template <bool RELOC>
__global__ void __launch_bounds__(THREADS, 1)
    seg_paged_one_kernel(const __grid_constant__ Args a, const __grid_constant__ Maps mp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  const tt::Ctx c{bar, reinterpret_cast<volatile uint32_t*>(misc + 1), a.status};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Tile t = a.tiles[blockIdx.x];
  const Req rq = a.reqs[t.req];
  const int nb = t.je - t.jb;  // this CTA's walk steps

  if (tid == 0) {
    for (int i = 0; i < RING; ++i) {
      tc::mbar_init(&bar[B_FULL + i], 1);
      tc::mbar_init(&bar[B_EMPTY + i], 1);
    }
    tc::mbar_init(&bar[B_QFULL], 8);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bar[B_SFULL + b], 1);
      tc::mbar_init(&bar[B_SFREE + b], 8);
    }
    tc::mbar_init(&bar[B_PREADY], 8);
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
      tc::prefetch_tmap(&mp.k);
      tc::prefetch_tmap(&mp.v);
      const int32_t* tab = a.table + rq.table_off + int64_t(t.g) * a.max_blocks;
      uint32_t cnt = 0;
      bool ok = true;
      auto load = [&](const CUtensorMap* map, int page) {
        const int slot = cnt % RING;
        if (!tt::wait_bar(c, B_EMPTY + slot, ((cnt / RING) & 1) ^ 1)) return false;
        tc::mbar_arrive_expect_tx(&bar[B_FULL + slot], SLOT);
        tc::tma_load_4d(smem_u32(sm + OFF_RING + slot * SLOT), map, &bar[B_FULL + slot], 0, 0, 0,
                        page);
        ++cnt;
        return true;
      };
      // K_j, then V_{j-1}: the order in which the issuer consumes them
      for (int j = 0; j <= nb && ok; ++j) {
        if (j < nb) ok = load(&mp.k, tab[block_of(t, t.jb + j)]);
        if (ok && j >= 1) ok = load(&mp.v, tab[block_of(t, t.jb + j - 1)]);
      }
      // copies in flight land before the CTA may exit
      for (uint32_t k = (cnt > RING ? cnt - RING : 0); k < cnt; ++k)
        tt::drain_bar(c, B_FULL + k % RING, (k / RING) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      bool ok = tt::wait_bar(c, B_QFULL, 0);
      tc::tc_fence_after();
      const uint32_t idS = tc::idesc_bf16(128, 128, false, false);
      const uint32_t idPV = tc::idesc_bf16(128, 128, false, true);
      const uint32_t ra = smem_u32(sm + OFF_RING);
      // relocated documents, tiles of at most 64 pairs in use (memory-bound
      // decode and tail tiles): P enters P.V as bf16 hi + lo parts
      const bool psplit = RELOC && t.rows * a.G <= 64;
      uint32_t cnt = 0;
      auto pv = [&](int jj) {
        if (!tt::wait_bar(c, B_PREADY, jj & 1)) return false;
        tc::tc_fence_after();
        const int slot = cnt % RING;
        if (!tt::wait_bar(c, B_FULL + slot, (cnt / RING) & 1)) return false;
        tc::tc_fence_after();
        const uint32_t base = ra + slot * SLOT;
        const uint32_t tp = RELOC ? T_S + 128 * (jj & 1) : T_P;
        // B = V[16 keys x 128 dims]: two 64-dim chunks 16 KB apart (LBO)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tc::mma_ts(tbase + T_O, tbase + tp + 8 * k, tc::sdesc_sw128(base + 2048 * k, CHUNK, 1024),
                     idPV, (jj > 0 || k > 0) ? 1u : 0u);
        if (psplit) {
          // the lo part of P: half h of the keys at columns 64 + 32 h of the
          // buffer, keys 32..63 of the half before keys 0..31
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t lc = 64 + 32 * (k >> 2) + (((k >> 1) & 1) ? 0 : 16) + 8 * (k & 1);
            tc::mma_ts(tbase + T_O, tbase + tp + lc, tc::sdesc_sw128(base + 2048 * k, CHUNK, 1024),
                       idPV, 1u);
          }
        }
        tc::mma_commit(&bar[B_EMPTY + slot]);
        ++cnt;
        tc::mma_commit(&bar[B_ODONE]);
        return true;
      };
      uint32_t qph = 1;        // query phases consumed (the first above)
      int32_t cs_prev = -1;    // relocated documents: offset index of the last step
      for (int j = 0; j < nb && ok; ++j) {
        const int b = j & 1;
        ok = tt::wait_bar(c, B_SFREE + b, ((j >> 1) & 1) ^ 1);
        if (!ok) break;
        int32_t csj = 0;
        if (RELOC) {
          // a new offset: the lanes rewrite R(-delta) q once S of the last
          // step is done (no S MMA still reads the old query)
          csj = cs_of(a, t, rq, j);
          if (j > 0 && csj != cs_prev) ok = tt::wait_bar(c, B_QFULL, qph++ & 1);
          cs_prev = csj;
          if (!ok) break;
        }
        tc::tc_fence_after();
        const int slot = cnt % RING;
        ok = tt::wait_bar(c, B_FULL + slot, (cnt / RING) & 1);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t base = ra + slot * SLOT;
        // A = Q[128 rows x 16 dims] from tensor memory (8 columns per step);
        // relocated documents: the hi part, then (offset not zero) the lo part
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_ts(tbase + T_S + 128 * b, tbase + (RELOC ? T_QH : T_Q) + 8 * (4 * cc + k),
                       tc::sdesc_sw128(base + cc * CHUNK + 32 * k, 16, 1024), idS, (cc | k) != 0);
        if (RELOC && csj != 0) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc::mma_ts(tbase + T_S + 128 * b, tbase + T_QL + 8 * (4 * cc + k),
                         tc::sdesc_sw128(base + cc * CHUNK + 32 * k, 16, 1024), idS, 1);
        }
        tc::mma_commit(&bar[B_EMPTY + slot]);
        ++cnt;
        tc::mma_commit(&bar[B_SFULL + b]);
        if (j >= 1) ok = pv(j - 1);
      }
      if (ok && nb > 0) pv(nb - 1);
      tc::mma_commit(&bar[B_FINAL]);
    }
  } else {
    // ------------------------------------------- softmax and epilogue ----
    const int lw = warp - 2;           // 0..7
    const int hf = lw >> 2;            // half of the keys and of the output columns
    const int quarter = warp & 3;      // TMEM lane quarter this warp may access
    const int m = quarter * 32 + lane;
    const int lid = lw * 32 + lane;    // 0..255
    const int r = m / a.G, h = m - r * a.G;
    const int p = t.p0 + r;
    const bool valid = r < t.rows;
    const bool glob = a.role[t.g] != 0;
    const uint32_t lt = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    const int sink = a.sink, window = a.window;
    const int64_t row = rq.row_base + (p - rq.q_row_begin);
    const int head = t.g * a.G + h;
    const bool psplit = RELOC && t.rows * a.G <= 64;  // P.V with P as hi + lo (see the issuer)
    float* xmax = reinterpret_cast<float*>(sm + OFF_X);          // [2][2][128]
    float* xsum = xmax + 4 * 128;                                 // [2][128]
    // this thread's half of the query row (dims 64 hf .. 64 hf + 63) ->
    // tensor memory, 32-bit column c = dims 2c, 2c + 1 (A operand of the
    // score MMAs); rows past the request's end are zero
    uint32_t qw[32];
    {
      const uint4* src = valid ? reinterpret_cast<const uint4*>(a.q + (row * a.Hq + head) * DH) + 8 * hf
                               : nullptr;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 v = src ? __ldg(src + u) : make_uint4(0, 0, 0, 0);
        qw[4 * u] = v.x;
        qw[4 * u + 1] = v.y;
        qw[4 * u + 2] = v.z;
        qw[4 * u + 3] = v.w;
      }
    }
    // relocated documents: R(-delta) q for the offset with index ci (RedKnot
    // blog, "Insight 1"; the query turns instead of the cached keys), this
    // thread's 32 rotation pairs (pair 32 hf + i: dims 2i, 2i + 1 of its
    // half), as bf16 hi and lo parts
    auto put_q = [&](int32_t ci) {
      if (RELOC) {
        const float4* cs4 = reinterpret_cast<const float4*>(a.cs + int64_t(ci) * 128 + 64 * hf);
        // two passes (hi, then lo) keep one 32-word array live at a time
#pragma unroll 1
        for (int part = 0; part < 2; ++part) {
          uint32_t w32[32];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const float4 w = __ldg(cs4 + u);  // (cos, sin) of pairs 2u, 2u + 1 of the half
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int i = 2 * u + e;
              const float co = e ? w.z : w.x, si = e ? w.w : w.y;
              const float x = __uint_as_float(qw[i] << 16), y = __uint_as_float(qw[i] & 0xffff0000u);
              const float xr = fmaf(x, co, y * si), yr = fmaf(-x, si, y * co);
              const uint32_t hw = pack_bf16x2(xr, yr);
              w32[i] = part == 0 ? hw
                                 : pack_bf16x2(xr - __uint_as_float(hw << 16),
                                               yr - __uint_as_float(hw & 0xffff0000u));
            }
          }
          tc::tmem_st32(lt + (part == 0 ? T_QH : T_QL) + 32 * hf, w32);
        }
      } else {
        tc::tmem_st32(lt + T_Q + 32 * hf, qw);
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[B_QFULL]);
    };
    put_q(RELOC && nb > 0 ? cs_of(a, t, rq, 0) : 0);
    float m_run = -INFINITY, l_run = 0.f;
    bool okw = true;
    for (int j = 0; j < nb; ++j) {
      const int b = j & 1;
      const int k0 = block_of(t, t.jb + j) * PAGE + 64 * hf;  // this thread's 64 keys
      if (okw) okw = __all_sync(0xffffffffu, tt::wait_bar(c, B_SFULL + b, (j >> 1) & 1));
      uint32_t s[2][32];
      float mx = -INFINITY;
      if (okw) {
        tc::tc_fence_after();
        tc::tmem_ld32(lt + T_S + 128 * b + 64 * hf, s[0]);
        tc::tmem_ld32(lt + T_S + 128 * b + 64 * hf + 32, s[1]);
        tc::tmem_wait_ld();
        // S of this step is done, so no S MMA reads the query any more: a
        // new offset at the next step gets its R(-delta) q now (the issuer
        // waits for it before the next S)
        if (RELOC && j + 1 < nb) {
          const int32_t cn = cs_of(a, t, rq, j + 1);
          if (cn != cs_of(a, t, rq, j)) put_q(cn);
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar[B_SFREE + b]);
        // every key of this half block visible for this row?  (then no masks)
        const bool full = valid && k0 + 63 <= p && (glob || k0 >= p - window || k0 + 64 <= sink);
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (__all_sync(0xffffffffu, full)) {
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2)
#pragma unroll
            for (int i = 0; i < 32; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(s[q2][i]));
        } else {
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int key = k0 + 32 * q2 + i;
              bool vis = valid && key <= p;
              if (!glob) vis = vis && (key < sink || key >= p - window);
              const float x = vis ? __uint_as_float(s[q2][i]) : -INFINITY;
              s[q2][i] = __float_as_uint(x);
              mx4[i & 3] = fmaxf(mx4[i & 3], x);
            }
          }
        }
        mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
        xmax[(b * 2 + hf) * 128 + m] = mx;
      }
      // every lane warp votes each block: the halves exchange their maxima,
      // and a failed wait anywhere makes all of them leave together
      if (!tc::named_and(2, 256, okw)) {
        okw = false;
        break;
      }
      mx = fmaxf(mx, xmax[(b * 2 + (hf ^ 1)) * 128 + m]);
      bool need = false;
      float alpha = 1.f;
      if (mx > m_run + 8.f) {  // lazy rescale: only when the max grows by more than 2^8
        if (m_run != -INFINITY) {
          need = true;
          alpha = fast_exp2(m_run - mx);
        }
        m_run = mx;
      }
      const float nbias = (m_run == -INFINITY) ? 0.f : -m_run;
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};
      // P in place: keys 2i, 2i + 1 of column block q2 go to word 16 q2 + i;
      // relocated documents also keep the lo parts P - bf16(P): those of
      // column block 1 in s[1][i] (already read), those of block 0 in lo0
      // and then s[1][16 + i]
      uint32_t lo0[16];
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(s[q2][2 * i]), sl2, nbias));
          const float p1 = fast_exp2(fmaf(__uint_as_float(s[q2][2 * i + 1]), sl2, nbias));
          ls4[i & 3] += p0 + p1;
          const uint32_t hw = pack_bf16x2(p0, p1);
          s[0][16 * q2 + i] = hw;
          if (RELOC) {
            const uint32_t lw =
                pack_bf16x2(p0 - __uint_as_float(hw << 16), p1 - __uint_as_float(hw & 0xffff0000u));
            if (q2 == 0)
              lo0[i] = lw;
            else
              s[1][i] = lw;
          }
        }
      }
      if (RELOC) {
#pragma unroll
        for (int i = 0; i < 16; ++i) s[1][16 + i] = lo0[i];
      }
      l_run = l_run * alpha + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
      // the previous P.V must be done before P and O are touched
      if (j >= 1) okw = __all_sync(0xffffffffu, tt::wait_bar(c, B_ODONE, (j - 1) & 1));
      if (okw) {
        tc::tc_fence_after();
        tc::tmem_st32(lt + (RELOC ? T_S + 128 * b : T_P) + 32 * hf, s[0]);
        if (psplit) tc::tmem_st32(lt + T_S + 128 * b + 64 + 32 * hf, s[1]);
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int q8 = 0; q8 < 2; ++q8) {
            uint32_t o[32];
            tc::tmem_ld32(lt + T_O + 64 * hf + 32 * q8, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tc::tmem_st32(lt + T_O + 64 * hf + 32 * q8, o);
          }
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar[B_PREADY]);
      }
    }
    // ---- epilogue ----
    bool ok = okw;
    if (ok) ok = __all_sync(0xffffffffu, tt::wait_bar(c, B_FINAL, 0));
    tc::tc_fence_after();
    xsum[hf * 128 + m] = l_run;
    ok = tc::named_and(3, 256, ok);  // every lane warp; also publishes the sums
    const float l_tot = l_run + xsum[(hf ^ 1) * 128 + m];
    if (t.nparts > 1) {
      if (ok) {
        const int nl = t.rows * a.G;  // lanes in use
        const int64_t slot = int64_t(t.lane0) + int64_t(t.part - t.part_first) * nl + m;
        const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
        float4* w4 = valid ? reinterpret_cast<float4*>(a.ws_o + slot * DH + 64 * hf) : nullptr;
        // tcgen05.ld is warp-aligned: every lane loads, only the used ones store
#pragma unroll 1
        for (int q8 = 0; q8 < 2; ++q8) {
          uint32_t o[32];
          tc::tmem_ld32(lt + T_O + 64 * hf + 32 * q8, o);
          tc::tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
              w4[8 * q8 + u] = make_float4(__uint_as_float(o[4 * u]) * inv, __uint_as_float(o[4 * u + 1]) * inv,
                                           __uint_as_float(o[4 * u + 2]) * inv, __uint_as_float(o[4 * u + 3]) * inv);
          }
        }
        if (valid && hf == 0)
          a.ws_lse[slot] = l_tot > 0.f ? m_run * 0.6931471805599453f + logf(l_tot) : -INFINITY;
        __threadfence();
        tc::named_sync(1, 256);
        volatile int* last = reinterpret_cast<volatile int*>(misc + 2);
        if (lid == 0) *last = atomicAdd(a.ws_ticket + t.group, 1) == t.nparts - 1;
        tc::named_sync(1, 256);
        if (*last) {
          __threadfence();
          merge_parts(a, t, rq, lid, 256);
        }
      }
    } else if (ok) {
      const bool st = valid && l_tot > 0.f;
      const float inv = st ? 1.f / l_tot : 0.f;
      uint16_t* dst = st ? a.out + (row * a.Hq + head) * DH + 64 * hf : nullptr;
#pragma unroll 1
      for (int q8 = 0; q8 < 2; ++q8) {
        uint32_t o[32];
        tc::tmem_ld32(lt + T_O + 64 * hf + 32 * q8, o);
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
      if (st && hf == 0) a.lse[row * a.Hq + head] = m_run * 0.6931471805599453f + logf(l_tot);
    }
  }

  // ------------------------------------------------------------ teardown --
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tt::drain_bar(c, B_FINAL, 0);  // the MMA pipe is empty before TMEM is released
    tc::tc_fence_after();
    tc::tmem_dealloc(tbase, 512);
  }
}

}  // namespace one

// ---- tiles of at most 16 query pairs (decode steps) on mma.sync ------------
// A persistent kernel (one CTA per SM) walks the tile list with a stride of
// the grid, so the page ring stays full across tile boundaries.  The query
// pairs (row r, head h) -> pair r G + h sit on the 16-row side of the
// m16n8k16 tile, the keys on its 8-column side.  Warp 8 streams the K and V
// pages (32 KB boxes, chunk-major, 128-byte swizzled) through a six-slot
// ring; compute warp w (0..7) takes keys 16 w .. 16 w + 15 of every block:
// S = Q K^T on its 16 keys, its own online softmax, O += P V with P taken
// straight from the score fragments.  At the end of a tile the eight warps'
// partial states are merged through shared memory (log-sum-exp), eight pairs
// per pass; a split part leaves its normalised result in the workspace and
// the last part merges the parts.
namespace dec {

constexpr int CW = 8;                          // compute warps
constexpr int THREADS = 32 * (CW + 1);         // + the producer warp
constexpr int RING = 6;
constexpr uint32_t SLOT = 2 * CHUNK;           // one K or V page
constexpr uint32_t OFF_RING = 0;
constexpr uint32_t OFF_MERGE = OFF_RING + RING * SLOT;   // [CW][8 pairs][128] fp32
constexpr uint32_t OFF_ML = OFF_MERGE + CW * 8 * DH * 4;  // m [CW][16], l [CW][16]
constexpr uint32_t OFF_BAR = OFF_ML + 2 * CW * 16 * 4;
enum { B_FULL = 0, B_EMPTY = RING, NBAR = 2 * RING };
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
static_assert(OFF_MERGE % 16 == 0 && OFF_ML % 16 == 0 && OFF_BAR % 8 == 0, "alignment");

__device__ __forceinline__ uint32_t ldg32(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint32_t*>(p));
}

__global__ void __launch_bounds__(THREADS, 1)
    seg_paged_dec_kernel(const __grid_constant__ Args a, const __grid_constant__ Maps mp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  const tt::Ctx c{bar, reinterpret_cast<volatile uint32_t*>(misc + 1), a.status};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < RING; ++i) {
      tc::mbar_init(&bar[B_FULL + i], 1);
      tc::mbar_init(&bar[B_EMPTY + i], CW);
    }
    misc[1] = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();

  if (warp == CW) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      tc::prefetch_tmap(&mp.k);
      tc::prefetch_tmap(&mp.v);
      uint32_t cnt = 0;
      bool ok = true;
      auto load = [&](const CUtensorMap* map, int page) {
        const int slot = cnt % RING;
        if (!tt::wait_bar(c, B_EMPTY + slot, ((cnt / RING) & 1) ^ 1)) return false;
        tc::mbar_arrive_expect_tx(&bar[B_FULL + slot], SLOT);
        tc::tma_load_4d(smem_u32(sm + OFF_RING + slot * SLOT), map, &bar[B_FULL + slot], 0, 0, 0,
                        page);
        ++cnt;
        return true;
      };
      for (int ti = blockIdx.x; ti < a.num_tiles && ok; ti += gridDim.x) {
        const Tile t = a.tiles[ti];
        const int32_t* tab = a.table + a.reqs[t.req].table_off + int64_t(t.g) * a.max_blocks;
        for (int j = t.jb; j < t.je && ok; ++j) {
          const int page = tab[block_of(t, j)];
          ok = load(&mp.k, page) && load(&mp.v, page);
        }
      }
      // copies in flight land before the CTA may exit
      for (uint32_t k = (cnt > RING ? cnt - RING : 0); k < cnt; ++k)
        tt::drain_bar(c, B_FULL + k % RING, (k / RING) & 1);
    }
  } else {
    // --------------------------------------------------- compute warps ---
    const int g8 = lane >> 2, t4 = lane & 3;
    const uint32_t ring = smem_u32(sm + OFF_RING);
    float* mbuf = reinterpret_cast<float*>(sm + OFF_MERGE);  // [CW][8][DH]
    float* mlm = reinterpret_cast<float*>(sm + OFF_ML);      // [CW][16]
    float* mll = mlm + CW * 16;                              // [CW][16]
    const float sl2 = a.scale_log2;
    const int sink = a.sink, window = a.window;
    // ldmatrix row addresses of this lane (matrix lane >> 3, row lane & 7):
    // scores read K rows 16 warp + 8 ((lane >> 3) >> 1) + (lane & 7) at
    // dim unit (lane >> 3) & 1 of a k-step; P.V reads V rows
    // 16 warp + 8 ((lane >> 3) & 1) + (lane & 7) at dim unit (lane >> 3) >> 1
    const int mi = lane >> 3;
    const uint32_t krow = 16 * warp + 8 * (mi >> 1) + (lane & 7);
    const uint32_t vrow = 16 * warp + 8 * (mi & 1) + (lane & 7);
    uint32_t cnt = 0;
    bool ok = true;
    for (int ti = blockIdx.x; ti < a.num_tiles; ti += gridDim.x) {
      const Tile t = a.tiles[ti];
      const Req rq = a.reqs[t.req];
      const bool glob = a.role[t.g] != 0;
      const int np = t.rows * a.G;  // pairs in use (<= 16)
      // this lane's two pairs: rows g8 and g8 + 8 of the fragments
      int pp[2];
      bool pv[2];
      uint32_t qa[8][4];
      {
        const uint16_t* qr[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int n = g8 + 8 * e;
          const int r = n / a.G, h = n - r * a.G;
          pv[e] = n < np;
          pp[e] = t.p0 + r;
          const int64_t row = rq.row_base + (pp[e] - rq.q_row_begin);
          qr[e] = pv[e] ? a.q + (row * a.Hq + t.g * a.G + h) * DH : nullptr;
        }
        // A fragments of Q: k-step kk covers dims 16 kk .. 16 kk + 15
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int d = 16 * kk + 2 * t4;
          qa[kk][0] = qr[0] ? ldg32(qr[0] + d) : 0u;
          qa[kk][1] = qr[1] ? ldg32(qr[1] + d) : 0u;
          qa[kk][2] = qr[0] ? ldg32(qr[0] + d + 8) : 0u;
          qa[kk][3] = qr[1] ? ldg32(qr[1] + d + 8) : 0u;
        }
      }
      float o[16][4];
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

      for (int j = t.jb; j < t.je && ok; ++j) {
        const int kb = block_of(t, j) * PAGE;
        // ---- S = Q K^T on this warp's 16 keys ----
        int slot = cnt % RING;
        ok = __all_sync(0xffffffffu, tt::wait_bar(c, B_FULL + slot, (cnt / RING) & 1));
        if (!ok) break;
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const uint32_t base = ring + slot * SLOT + krow * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t unit = 2 * (kk & 3) + (mi & 1);
            uint32_t b[4];
            ldsm_x4(b, base + (kk >> 2) * CHUNK + ((unit ^ (krow & 7)) << 4));
            mma16816(s[0], qa[kk], b[0], b[1]);
            mma16816(s[1], qa[kk], b[2], b[3]);
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar[B_EMPTY + slot]);
        ++cnt;
        // ---- mask, online softmax (log2 domain) ----
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int key = kb + 16 * warp + 8 * nt + 2 * t4 + u;
              bool vis = pv[e] && key <= pp[e];
              if (!glob) vis = vis && (key < sink || key >= pp[e] - window);
              const float x = vis ? s[nt][2 * e + u] * sl2 : -INFINITY;
              s[nt][2 * e + u] = x;
              mx[e] = fmaxf(mx[e], x);
            }
        float alpha[2], nb[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 1));
          mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 2));
          const float mn = fmaxf(m_run[e], mx[e]);
          alpha[e] = (m_run[e] == -INFINITY) ? 1.f : fast_exp2(m_run[e] - mn);
          nb[e] = (mn == -INFINITY) ? 0.f : -mn;
          m_run[e] = mn;
        }
        uint32_t pa[4];
        float ls[2] = {0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float p0 = fast_exp2(s[nt][2 * e] + nb[e]);
            const float p1 = fast_exp2(s[nt][2 * e + 1] + nb[e]);
            ls[e] += p0 + p1;
            pa[2 * nt + e] = pack_bf16x2(p0, p1);
          }
#pragma unroll
        for (int e = 0; e < 2; ++e) l_run[e] = l_run[e] * alpha[e] + ls[e];
        if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            o[i][0] *= alpha[0];
            o[i][1] *= alpha[0];
            o[i][2] *= alpha[1];
            o[i][3] *= alpha[1];
          }
        }
        // ---- O += P V on this warp's 16 keys ----
        slot = cnt % RING;
        ok = __all_sync(0xffffffffu, tt::wait_bar(c, B_FULL + slot, (cnt / RING) & 1));
        if (!ok) break;
        {
          const uint32_t base = ring + slot * SLOT + vrow * 128;
#pragma unroll
          for (int d2 = 0; d2 < 8; ++d2) {
            const uint32_t unit = 2 * (d2 & 3) + (mi >> 1);
            uint32_t b[4];
            ldsm_x4_t(b, base + (d2 >> 2) * CHUNK + ((unit ^ (vrow & 7)) << 4));
            mma16816(o[2 * d2], pa, b[0], b[1]);
            mma16816(o[2 * d2 + 1], pa, b[2], b[3]);
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar[B_EMPTY + slot]);
        ++cnt;
      }
      // every compute warp agrees before the merge (a failed wait anywhere
      // makes all of them leave the tile loop together)
      ok = tc::named_and(1, 32 * CW, ok);
      if (!ok) break;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 1);
        l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 2);
      }
      const bool split = t.nparts > 1;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if (e == 1 && np <= 8) break;
        // this warp's state of pairs 8 e .. 8 e + 7
#pragma unroll
        for (int i = 0; i < 16; ++i)
          *reinterpret_cast<float2*>(mbuf + (warp * 8 + g8) * DH + 8 * i + 2 * t4) =
              make_float2(o[i][2 * e], o[i][2 * e + 1]);
        if (t4 == 0) {
          mlm[warp * 16 + g8 + 8 * e] = m_run[e];
          mll[warp * 16 + g8 + 8 * e] = l_run[e];
        }
        tc::named_sync(1, 32 * CW);
        {
          const int n = 8 * e + (tid >> 5), d0 = 4 * (tid & 31);
          if (n < np) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < CW; ++w) M = fmaxf(M, mlm[w * 16 + n]);
            float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < CW; ++w) {
              const float mw = mlm[w * 16 + n];
              const float wt = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
              L += wt * mll[w * 16 + n];
              const float4 x = *reinterpret_cast<const float4*>(mbuf + (w * 8 + (n & 7)) * DH + d0);
              acc[0] += wt * x.x;
              acc[1] += wt * x.y;
              acc[2] += wt * x.z;
              acc[3] += wt * x.w;
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const float lse = L > 0.f ? M * 0.6931471805599453f + logf(L) : -INFINITY;
            const int r = n / a.G, h = n - r * a.G;
            if (split) {
              const int64_t sl = int64_t(t.lane0) + int64_t(t.part - t.part_first) * np + n;
              *reinterpret_cast<float4*>(a.ws_o + sl * DH + d0) =
                  make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
              if (d0 == 0) a.ws_lse[sl] = lse;
            } else if (L > 0.f) {
              const int64_t row = rq.row_base + (t.p0 + r - rq.q_row_begin);
              const int64_t oi = row * a.Hq + t.g * a.G + h;
              *reinterpret_cast<uint2*>(a.out + oi * DH + d0) =
                  make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                             pack_bf16x2(acc[2] * inv, acc[3] * inv));
              if (d0 == 0) a.lse[oi] = lse;
            }
          }
        }
        tc::named_sync(1, 32 * CW);  // the buffer is free for the next pass or tile
      }
      if (split) {
        __threadfence();
        volatile int* last = reinterpret_cast<volatile int*>(misc + 2);
        if (tid == 0) *last = atomicAdd(a.ws_ticket + t.group, 1) == t.nparts - 1;
        tc::named_sync(1, 32 * CW);
        const bool im_last = *last != 0;
        tc::named_sync(1, 32 * CW);  // the flag is read before the next tile may set it
        if (im_last) {
          __threadfence();
          merge_parts(a, t, rq, tid, 32 * CW);
        }
      }
    }
  }
  __syncthreads();
}

}  // namespace dec

}  // namespace sp
}  // namespace rk

struct rk_segpaged_plan_s {
  int device = -1;
  bool host_only = false;
  int32_t Hq = 0, Hkv = 0, G = 0, sink = 0, window = 0, max_blocks = 0;
  float scale = 0.f;
  int64_t num_pages = 0, rows = 0;
  int64_t split_lanes = 0, split_tiles = 0;
  size_t workspace_bytes = 0;
  rk_segpaged_info_t info{};
  std::vector<rk::sp::Req> reqs;
  std::vector<rk::sp::Tile> tiles;      // two sub-tiles per CTA
  std::vector<rk::sp::Tile> tiles_one;  // one sub-tile per CTA (<= 64 pairs in use)
  std::vector<rk::sp::Tile> tiles_dec;  // <= 16 pairs in use (decode steps), persistent kernel
  int32_t num_sms = 0;
  std::vector<int32_t> table;
  std::vector<uint8_t> role;
  bool reloc = false;             // relocated documents: every tile on the one-sub-tile kernel
  std::vector<int32_t> blk_cs;    // [R][max_blocks] offset index of each block
  std::vector<float> cs;          // [offsets][64][2] cos, sin of delta * theta_j
  int32_t* d_blk_cs = nullptr;
  float* d_cs = nullptr;
  rk::sp::Req* d_reqs = nullptr;
  rk::sp::Tile* d_tiles = nullptr;
  rk::sp::Tile* d_tiles_one = nullptr;
  rk::sp::Tile* d_tiles_dec = nullptr;
  int32_t* d_table = nullptr;
  uint8_t* d_role = nullptr;
  int32_t* d_status = nullptr;
};

namespace {

using rk::sp::PAGE;
constexpr int kSplitBlocks = 32;  // walk steps per part of a split tile (<= 64 pairs)
constexpr int kDecSplit = 32;     // walk steps per part of a split tile of <= 16 pairs

void sp_free(rk_segpaged_plan_s* p) {
  cudaFree(p->d_reqs);
  cudaFree(p->d_tiles);
  cudaFree(p->d_tiles_one);
  cudaFree(p->d_tiles_dec);
  cudaFree(p->d_table);
  cudaFree(p->d_role);
  cudaFree(p->d_status);
  cudaFree(p->d_blk_cs);
  cudaFree(p->d_cs);
  p->d_blk_cs = nullptr;
  p->d_cs = nullptr;
  p->d_reqs = nullptr;
  p->d_tiles = nullptr;
  p->d_tiles_one = nullptr;
  p->d_tiles_dec = nullptr;
  p->d_table = nullptr;
  p->d_role = nullptr;
  p->d_status = nullptr;
}

template <typename T>
rk_status_t sp_upload(const std::vector<T>& v, T** dptr, cudaStream_t s) {
  *dptr = nullptr;
  if (v.empty()) return RK_OK;
  if (cudaMalloc(reinterpret_cast<void**>(dptr), v.size() * sizeof(T)) != cudaSuccess) {
    *dptr = nullptr;
    return RK_ERR_CUDA;
  }
  return cudaMemcpyAsync(*dptr, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice, s) ==
                 cudaSuccess
             ? RK_OK
             : RK_ERR_CUDA;
}

// keys a Local row p sees: [0, min(sink, p + 1)) u [max(0, p - w), p]
int64_t local_keys(int64_t p, int64_t sink, int64_t window) {
  const int64_t lo = std::max<int64_t>(0, p - window);
  if (lo <= sink) return p + 1;
  return std::min<int64_t>(sink, p + 1) + (p - lo + 1);
}

rk_status_t sp_build(const rk_segpaged_desc_t* d, rk_segpaged_plan_s* p) {
  if (!d->seq_len || !d->q_row_begin || !d->block_table || !d->kv_head_role) return RK_ERR_NULL;
  const int R = d->num_requests;
  if (R < 1 || d->num_kv_heads < 1 || d->num_q_heads < 1 || d->num_q_heads % d->num_kv_heads)
    return RK_ERR_INVALID_ARG;
  const int G = d->num_q_heads / d->num_kv_heads;
  if (d->head_dim != rk::sp::DH || d->page_size != PAGE ||
      !(G == 1 || G == 2 || G == 4 || G == 8 || G == 16))
    return RK_ERR_UNSUPPORTED_DIMS;
  if (d->num_pages < 1 || d->max_blocks < 1 || d->sink < 0 || d->window < 0)
    return RK_ERR_INVALID_ARG;
  if (!(d->softmax_scale > 0.f) || !std::isfinite(d->softmax_scale)) return RK_ERR_INVALID_ARG;
  if (d->flags & ~(RK_SEGPAGED_HOST_ONLY | RK_SEGPAGED_DENSE_MASK)) return RK_ERR_INVALID_ARG;
  if (d->num_pages > INT32_MAX || int64_t(d->num_q_heads) * 256 > INT32_MAX)
    return RK_ERR_CAPACITY;
  const int Hkv = d->num_kv_heads;
  for (int g = 0; g < Hkv; ++g)
    if (d->kv_head_role[g] > 1) return RK_ERR_INVALID_ARG;
  const bool dense = (d->flags & RK_SEGPAGED_DENSE_MASK) != 0;
  // relocated documents: one sub-tile of 128 / G rows per tile, every tile
  // on the one-sub-tile kernel (its query operand is R(-delta) q as hi + lo)
  const bool reloc = d->block_delta != nullptr;
  if (reloc && !(d->rope_base > 1.0) ) return RK_ERR_INVALID_ARG;
  const int RT = (reloc ? 128 : 256) / G;  // rows of a tile
  p->Hq = d->num_q_heads;
  p->Hkv = Hkv;
  p->G = G;
  p->sink = d->sink;
  p->window = d->window;
  p->max_blocks = d->max_blocks;
  p->scale = d->softmax_scale;
  p->num_pages = d->num_pages;
  p->host_only = (d->flags & RK_SEGPAGED_HOST_ONLY) != 0;
  p->role.assign(d->kv_head_role, d->kv_head_role + Hkv);
  const int64_t tab_n = int64_t(R) * Hkv * d->max_blocks;
  p->table.assign(d->block_table, d->block_table + tab_n);
  p->reloc = reloc;
  if (reloc) {
    // one cos / sin table per distinct offset (index 0: the zero offset),
    // angles in double precision: delta * base^(-2j / 128), j = 0..63
    std::map<int64_t, int32_t> index{{0, 0}};
    std::vector<int64_t> deltas{0};
    const int64_t nblk = int64_t(R) * d->max_blocks;
    p->blk_cs.resize(nblk);
    for (int64_t i = 0; i < nblk; ++i) {
      const int64_t dl = d->block_delta[i];
      if (dl < INT32_MIN || dl > INT32_MAX) return RK_ERR_INVALID_ARG;
      auto it = index.find(dl);
      if (it == index.end()) {
        if (deltas.size() >= (1u << 20)) return RK_ERR_CAPACITY;
        it = index.emplace(dl, static_cast<int32_t>(deltas.size())).first;
        deltas.push_back(dl);
      }
      p->blk_cs[i] = it->second;
    }
    p->cs.resize(deltas.size() * 128);
    for (size_t k = 0; k < deltas.size(); ++k)
      for (int j = 0; j < 64; ++j) {
        const double ang = double(deltas[k]) * std::pow(d->rope_base, -2.0 * j / 128.0);
        p->cs[k * 128 + 2 * j] = static_cast<float>(std::cos(ang));
        p->cs[k * 128 + 2 * j + 1] = static_cast<float>(std::sin(ang));
      }
  }
  rk_segpaged_info_t& info = p->info;
  info = rk_segpaged_info_t{};
  info.group = G;
  std::vector<std::pair<int64_t, rk::sp::Tile>> list, list_one, list_dec;
  int64_t rows = 0;
  for (int r = 0; r < R; ++r) {
    const int64_t T = d->seq_len[r], qb = d->q_row_begin[r];
    if (T < 1 || qb < 0 || qb >= T) return RK_ERR_INVALID_ARG;
    if (T > INT32_MAX - PAGE) return RK_ERR_CAPACITY;
    if ((T + PAGE - 1) / PAGE > d->max_blocks) return RK_ERR_INVALID_ARG;
    rk::sp::Req q{};
    q.T = static_cast<int32_t>(T);
    q.q_row_begin = static_cast<int32_t>(qb);
    q.row_base = rows;
    q.table_off = int64_t(r) * Hkv * d->max_blocks;
    q.blk_off = int64_t(r) * d->max_blocks;
    p->reqs.push_back(q);
    for (int64_t x = qb; x < T; ++x)
      for (int g = 0; g < Hkv; ++g)
        info.pairs += int64_t(G) * (d->kv_head_role[g] ? x + 1 : local_keys(x, d->sink, d->window));
    for (int g = 0; g < Hkv; ++g) {
      const int32_t* tab = d->block_table + q.table_off + int64_t(g) * d->max_blocks;
      const bool glob = d->kv_head_role[g] != 0;
      for (int64_t p0 = qb; p0 < T; p0 += RT) {
        rk::sp::Tile t{};
        t.req = r;
        t.g = g;
        t.p0 = static_cast<int32_t>(p0);
        t.rows = static_cast<int32_t>(std::min<int64_t>(RT, T - p0));
        const int64_t plast = p0 + t.rows - 1;
        t.hi = static_cast<int32_t>(plast / PAGE);
        t.sink_blocks = 0;
        t.win_lo = 0;
        if (!glob && !dense) {
          const int64_t lo = std::max<int64_t>(0, p0 - d->window);
          const int64_t lo_blk = lo / PAGE;
          const int64_t sink_blk = (std::min<int64_t>(d->sink, plast + 1) + PAGE - 1) / PAGE;
          if (lo_blk > sink_blk) {
            t.sink_blocks = static_cast<int32_t>(sink_blk);
            t.win_lo = static_cast<int32_t>(lo_blk);
          }
        }
        const int nb = t.sink_blocks + (t.hi - t.win_lo + 1);
        for (int j = 0; j < nb; ++j) {
          const int b = j < t.sink_blocks ? j : t.win_lo + (j - t.sink_blocks);
          if (tab[b] < 0 || tab[b] >= d->num_pages) return RK_ERR_INVALID_ARG;
        }
        info.kv_blocks += nb;
        // at most 16 pairs in use: decode kernel; at most 64 (or relocated
        // documents): one-sub-tile kernel
        const bool tiny = !reloc && t.rows * G <= 16;
        const bool small = reloc || t.rows * G <= 64;
        info.performed_pairs +=
            int64_t(nb) * (tiny ? 16 : (!reloc && t.rows > RT / 2) ? 256 : 128) * PAGE;
        t.jb = 0;
        t.je = nb;
        t.part = t.part_first = 0;
        t.nparts = 1;
        const int split_len = tiny ? kDecSplit : kSplitBlocks;
        if (small && t.rows * G <= 64 && nb > (tiny ? 3 * kDecSplit / 2 : 2 * kSplitBlocks)) {
          // a long walk of few rows: parts of split_len steps, merged at the end
          const int np = (nb + split_len - 1) / split_len;
          t.nparts = np;
          t.group = static_cast<int32_t>(p->split_tiles++);
          t.lane0 = static_cast<int32_t>(p->split_lanes);
          p->split_lanes += int64_t(np) * t.rows * G;
          info.split_parts += np;
          for (int q = 0; q < np; ++q) {
            rk::sp::Tile u = t;
            u.part = q;
            u.jb = q * split_len;
            u.je = std::min(nb, (q + 1) * split_len);
            (tiny ? list_dec : list_one).push_back({u.je - u.jb, u});
          }
          continue;
        }
        (tiny ? list_dec : small ? list_one : list).push_back({nb, t});
      }
    }
    rows += T - qb;
  }
  if (rows * d->num_q_heads > (int64_t(1) << 40) || list.size() > INT32_MAX / 2 ||
      list_one.size() > INT32_MAX / 2 || list_dec.size() > INT32_MAX / 2)
    return RK_ERR_CAPACITY;
  auto longest_first = [](const auto& x, const auto& y) { return x.first > y.first; };
  std::stable_sort(list.begin(), list.end(), longest_first);
  std::stable_sort(list_one.begin(), list_one.end(), longest_first);
  std::stable_sort(list_dec.begin(), list_dec.end(), longest_first);
  for (auto& e : list) p->tiles.push_back(e.second);
  for (auto& e : list_one) p->tiles_one.push_back(e.second);
  for (auto& e : list_dec) p->tiles_dec.push_back(e.second);
  p->rows = rows;
  info.rows = rows;
  info.tiles = static_cast<int64_t>(p->tiles.size() + p->tiles_one.size() + p->tiles_dec.size());
  if (p->split_lanes > INT32_MAX / 2 || p->split_tiles > INT32_MAX / 2) return RK_ERR_CAPACITY;
  if (p->split_tiles) {
    size_t b = static_cast<size_t>(p->split_lanes) * (rk::sp::DH + 1) * sizeof(float);
    b = (b + 255) & ~size_t(255);
    b += static_cast<size_t>(p->split_tiles) * sizeof(int32_t);
    p->workspace_bytes = (b + 255) & ~size_t(255);
  }
  return RK_OK;
}

}  // namespace

extern "C" rk_status_t rk_segpaged_plan(const rk_segpaged_desc_t* desc, void* stream,
                                        rk_segpaged_plan_t* out) {
  if (!out) return RK_ERR_NULL;
  *out = nullptr;
  if (!desc) return RK_ERR_NULL;
  rk_segpaged_plan_s* p = new (std::nothrow) rk_segpaged_plan_s();
  if (!p) return RK_ERR_CAPACITY;
  rk_status_t st = sp_build(desc, p);
  if (st == RK_OK && !p->host_only) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaGetDevice(&p->device) != cudaSuccess) st = RK_ERR_CUDA;
    if (st == RK_OK) st = sp_upload(p->reqs, &p->d_reqs, s);
    if (st == RK_OK) st = sp_upload(p->tiles, &p->d_tiles, s);
    if (st == RK_OK) st = sp_upload(p->tiles_one, &p->d_tiles_one, s);
    if (st == RK_OK) st = sp_upload(p->tiles_dec, &p->d_tiles_dec, s);
    if (st == RK_OK &&
        cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess)
      st = RK_ERR_CUDA;
    if (st == RK_OK) st = sp_upload(p->table, &p->d_table, s);
    if (st == RK_OK) st = sp_upload(p->role, &p->d_role, s);
    if (st == RK_OK) st = sp_upload(p->blk_cs, &p->d_blk_cs, s);
    if (st == RK_OK) st = sp_upload(p->cs, &p->d_cs, s);
    if (st == RK_OK) {
      if (cudaMalloc(reinterpret_cast<void**>(&p->d_status), sizeof(int32_t)) != cudaSuccess ||
          cudaMemsetAsync(p->d_status, 0, sizeof(int32_t), s) != cudaSuccess)
        st = RK_ERR_CUDA;
    }
    // the host vectors are pageable: the uploads complete before returning
    if (st == RK_OK && cudaStreamSynchronize(s) != cudaSuccess) st = RK_ERR_CUDA;
    if (st != RK_OK) sp_free(p);
  }
  if (st != RK_OK) {
    delete p;
    return st;
  }
  *out = p;
  return RK_OK;
}

extern "C" rk_status_t rk_segpaged_forward(rk_segpaged_plan_t p, const void* q, const void* k_pages,
                                           const void* v_pages, void* out, float* lse,
                                           void* workspace, size_t workspace_bytes,
                                           void* stream) {
  if (!p || !q || !k_pages || !v_pages || !out || !lse) return RK_ERR_NULL;
  if (p->host_only) return RK_ERR_PLAN_MISMATCH;
  auto mis = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) != 0; };
  if (mis(q) || mis(k_pages) || mis(v_pages) || mis(out) || (reinterpret_cast<uintptr_t>(lse) & 3))
    return RK_ERR_ALIGNMENT;
  if (p->workspace_bytes) {
    if (!workspace || workspace_bytes < p->workspace_bytes) return RK_ERR_WORKSPACE;
    if (mis(workspace)) return RK_ERR_ALIGNMENT;
  }
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return RK_ERR_CUDA;
  if (cur != p->device) return RK_ERR_PLAN_MISMATCH;
  if (p->tiles.empty() && p->tiles_one.empty() && p->tiles_dec.empty()) return RK_OK;
  rk::sp::Maps mp{};
  {
    // a page viewed as (64 dims, 128 tokens, 2 chunks, pages): one page per box
    const uint64_t dims[4] = {64, PAGE, 2, static_cast<uint64_t>(p->num_pages)};
    const uint64_t strides[3] = {256, 128, 256 * PAGE};
    const uint32_t box[4] = {64, PAGE, 2, 1};
    if (!rk::make_tmap_bf16(&mp.k, k_pages, 4, dims, strides, box) ||
        !rk::make_tmap_bf16(&mp.v, v_pages, 4, dims, strides, box))
      return RK_ERR_CUDA;
  }
  rk::sp::Args a{};
  a.q = static_cast<const uint16_t*>(q);
  a.tiles = p->d_tiles;
  a.reqs = p->d_reqs;
  a.table = p->d_table;
  a.role = p->d_role;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.status = p->d_status;
  a.Hq = p->Hq;
  a.G = p->G;
  a.max_blocks = p->max_blocks;
  a.sink = p->sink;
  a.window = p->window;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.blk_cs = p->d_blk_cs;
  a.cs = p->d_cs;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p->split_tiles) {
    char* w = static_cast<char*>(workspace);
    a.ws_o = reinterpret_cast<float*>(w);
    size_t off = static_cast<size_t>(p->split_lanes) * rk::sp::DH * sizeof(float);
    a.ws_lse = reinterpret_cast<float*>(w + off);
    off += static_cast<size_t>(p->split_lanes) * sizeof(float);
    off = (off + 255) & ~size_t(255);
    a.ws_ticket = reinterpret_cast<int32_t*>(w + off);
    if (cudaMemsetAsync(a.ws_ticket, 0, static_cast<size_t>(p->split_tiles) * sizeof(int32_t), s) !=
        cudaSuccess)
      return RK_ERR_CUDA;
  }
  if (!p->tiles.empty()) {
    namespace k2 = rk::sp::two;
    if (cudaFuncSetAttribute(k2::seg_paged_two_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(k2::SMEM_BYTES)) != cudaSuccess)
      return RK_ERR_CUDA;
    a.tiles = p->d_tiles;
    k2::seg_paged_two_kernel<<<static_cast<unsigned>(p->tiles.size()), k2::THREADS, k2::SMEM_BYTES,
                               s>>>(a, mp);
    if (cudaGetLastError() != cudaSuccess) return RK_ERR_CUDA;
  }
  if (!p->tiles_one.empty()) {
    namespace k1 = rk::sp::one;
    auto kern = p->reloc ? k1::seg_paged_one_kernel<true> : k1::seg_paged_one_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(k1::SMEM_BYTES)) != cudaSuccess)
      return RK_ERR_CUDA;
    a.tiles = p->d_tiles_one;
    kern<<<static_cast<unsigned>(p->tiles_one.size()), k1::THREADS, k1::SMEM_BYTES, s>>>(a, mp);
    if (cudaGetLastError() != cudaSuccess) return RK_ERR_CUDA;
  }
  if (!p->tiles_dec.empty()) {
    namespace kd = rk::sp::dec;
    if (cudaFuncSetAttribute(kd::seg_paged_dec_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kd::SMEM_BYTES)) != cudaSuccess)
      return RK_ERR_CUDA;
    a.tiles = p->d_tiles_dec;
    a.num_tiles = static_cast<int32_t>(p->tiles_dec.size());
    // persistent: one CTA per SM strides over the tiles (longest first)
    const int grid = std::max(1, std::min<int>(a.num_tiles, p->num_sms));
    kd::seg_paged_dec_kernel<<<static_cast<unsigned>(grid), kd::THREADS, kd::SMEM_BYTES, s>>>(a, mp);
    if (cudaGetLastError() != cudaSuccess) return RK_ERR_CUDA;
  }
  return RK_OK;
}

extern "C" size_t rk_segpaged_workspace_bytes(rk_segpaged_plan_t p) {
  return p ? p->workspace_bytes : 0;
}

extern "C" rk_status_t rk_segpaged_plan_info(rk_segpaged_plan_t p, rk_segpaged_info_t* info) {
  if (!p || !info) return RK_ERR_NULL;
  *info = p->info;
  return RK_OK;
}

extern "C" rk_status_t rk_segpaged_last_device_status(rk_segpaged_plan_t p, void* stream) {
  if (!p) return RK_ERR_NULL;
  if (p->host_only) return RK_ERR_PLAN_MISMATCH;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, p->d_status, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemsetAsync(p->d_status, 0, sizeof(int32_t), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return RK_ERR_CUDA;
  return h ? static_cast<rk_status_t>(h) : RK_OK;
}

extern "C" void rk_segpaged_plan_destroy(rk_segpaged_plan_t p) {
  if (!p) return;
  if (!p->host_only) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device && p->device >= 0) cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    sp_free(p);
    if (cur != p->device && cur >= 0) cudaSetDevice(cur);
  }
  delete p;
}
