// SegPagedAttention for grouped-query attention on the tcgen05 path.
//
// RedKnot blog ("RedKnot, explained"), "Insight 3: savings must show up in
// memory": the KV cache is stored per KV head in pages; a Global head keeps
// the pages of the whole prompt, a Local head only those of its sink and
// window, so attention needs no mask over the prompt.  Visibility follows
// "Insight 1": Global heads see every k <= p, Local heads k <= p with
// k < sink or k >= p - w.
//
// A tile is 128 query pairs: 128 / G consecutive rows x the G query heads of
// one KV head, so each key page is read once for the whole group.  One CTA
// per tile (192 threads):
//   warp 0     TMA producer: for each key block its K page and, one block
//              behind, its V page (each a 32 KB box of 128 tokens x 128
//              dims, chunk-major, 128-byte swizzled) through a six-slot ring.
//   warp 1     MMA issuer: S_j = Q K_j^T (M = 128, N = 128 keys, A = Q and
//              B = K from shared memory) into one of two S buffers in tensor
//              memory, then O += P_{j-1} V_{j-1} (A = P from tensor memory,
//              B = V in MN-major form, N = 128).
//   warps 2-5  one thread per query pair (its TMEM lane): writes its query
//              row into shared memory (the A operand), masks the edge
//              blocks, keeps the running max in the log2 domain with a lazy
//              rescale of O when it grows by more than 2^8, writes P (bf16)
//              to tensor memory, and finally normalises and stores O and the
//              LSE.
// Tensor memory (512 columns): O (128) | S (2 x 128) | P (64, bf16 pairs).
// Every wait is bounded (2 s); on expiry the CTA records
// RK_ERR_DEVICE_TIMEOUT and every role stops; the producer waits (bounded)
// for its copies in flight and tensor memory is released after the MMA pipe
// has drained.

#include <algorithm>
#include <new>
#include <vector>

#include "rk_seg_paged.h"
#include "tc_tile.cuh"

namespace rk {
namespace sp {

constexpr int PAGE = 128;                   // tokens per page (= keys per block)
constexpr int DH = 128;                     // head dim
constexpr uint32_t CHUNK = 16384;           // 128 rows x 64 bf16
constexpr int THREADS = 192;
constexpr int RING = 6;
constexpr uint32_t SLOT = 2 * CHUNK;        // one K or V page
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_RING = 2 * CHUNK;
constexpr uint32_t OFF_BAR = OFF_RING + RING * SLOT;
enum {
  B_FULL = 0,
  B_EMPTY = RING,
  B_QFULL = 2 * RING,       // queries in shared memory (one arrival per lane warp)
  B_SFULL,                   // 2: S buffer j & 1 written
  B_SFREE = B_SFULL + 2,     // 2: S buffer read (one arrival per lane warp)
  B_PREADY = B_SFREE + 2,    // P_j written and O rescaled (one arrival per lane warp)
  B_ODONE,                   // O += P_j V_j done
  B_FINAL,
  NBAR
};
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
constexpr uint32_t T_O = 0, T_S = 128, T_P = 384;

struct Req {
  int32_t T;
  int32_t q_row_begin;
  int64_t row_base;      // first flattened row of the request
  int64_t table_off;     // offset of the request's [Hkv][max_blocks] block table
};

// 128 / G rows from p0 of KV head g; key blocks [0, sink_blocks) then
// [win_lo, hi] (sink_blocks = 0: [win_lo, hi] only).
struct Tile {
  int32_t req, g, p0, rows;
  int32_t sink_blocks, win_lo, hi, pad;
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
};

struct Maps {
  CUtensorMap k, v;
};

__device__ __forceinline__ int block_of(const Tile& t, int j) {
  return j < t.sink_blocks ? j : t.win_lo + (j - t.sink_blocks);
}

__global__ void __launch_bounds__(THREADS, 1)
    seg_paged_kernel(const __grid_constant__ Args a, const __grid_constant__ Maps mp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  const tt::Ctx c{bar, reinterpret_cast<volatile uint32_t*>(misc + 1), a.status};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Tile t = a.tiles[blockIdx.x];
  const Req rq = a.reqs[t.req];
  const int nb = t.sink_blocks + (t.hi - t.win_lo + 1);

  if (tid == 0) {
    for (int i = 0; i < RING; ++i) {
      tc::mbar_init(&bar[B_FULL + i], 1);
      tc::mbar_init(&bar[B_EMPTY + i], 1);
    }
    tc::mbar_init(&bar[B_QFULL], 4);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bar[B_SFULL + b], 1);
      tc::mbar_init(&bar[B_SFREE + b], 4);
    }
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
        if (j < nb) ok = load(&mp.k, tab[block_of(t, j)]);
        if (ok && j >= 1) ok = load(&mp.v, tab[block_of(t, j - 1)]);
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
      uint32_t cnt = 0;
      auto pv = [&](int jj) {
        if (!tt::wait_bar(c, B_PREADY, jj & 1)) return false;
        tc::tc_fence_after();
        const int slot = cnt % RING;
        if (!tt::wait_bar(c, B_FULL + slot, (cnt / RING) & 1)) return false;
        tc::tc_fence_after();
        const uint32_t base = ra + slot * SLOT;
        // B = V[16 keys x 128 dims]: two 64-dim chunks 16 KB apart (LBO)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tc::mma_ts(tbase + T_O, tbase + T_P + 8 * k, tc::sdesc_sw128(base + 2048 * k, CHUNK, 1024),
                     idPV, (jj > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(&bar[B_EMPTY + slot]);
        ++cnt;
        tc::mma_commit(&bar[B_ODONE]);
        return true;
      };
      for (int j = 0; j < nb && ok; ++j) {
        const int b = j & 1;
        ok = tt::wait_bar(c, B_SFREE + b, ((j >> 1) & 1) ^ 1);
        if (!ok) break;
        tc::tc_fence_after();
        const int slot = cnt % RING;
        ok = tt::wait_bar(c, B_FULL + slot, (cnt / RING) & 1);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t base = ra + slot * SLOT;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_ss(tbase + T_S + 128 * b, tc::sdesc_sw128(qa + cc * CHUNK + 32 * k, 16, 1024),
                       tc::sdesc_sw128(base + cc * CHUNK + 32 * k, 16, 1024), idS, (cc | k) != 0);
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
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const int r = m / a.G, h = m - r * a.G;
    const int p = t.p0 + r;
    const bool valid = r < t.rows;
    const bool glob = a.role[t.g] != 0;
    const uint32_t lt = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    const int sink = a.sink, window = a.window;
    const int64_t row = rq.row_base + (p - rq.q_row_begin);
    const int head = t.g * a.G + h;
    // this lane's query row -> shared memory: two 64-dim chunks of 128 rows,
    // 128-byte swizzle (A operand of the score MMAs); rows past the
    // request's end are zero
    {
      const uint4* src = valid ? reinterpret_cast<const uint4*>(a.q + (row * a.Hq + head) * DH)
                               : nullptr;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint4 v = src ? __ldg(src + u) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sm + OFF_Q + (u >> 3) * CHUNK + m * 128 +
                                  (((u & 7) ^ (m & 7)) << 4)) = v;
      }
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[B_QFULL]);
    }
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nb && ok; ++j) {
      const int b = j & 1;
      const int k0 = block_of(t, j) * PAGE;
      ok = __all_sync(0xffffffffu, tt::wait_bar(c, B_SFULL + b, (j >> 1) & 1));
      if (!ok) break;
      tc::tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tc::tmem_ld32(lt + T_S + 128 * b + 32 * q4, s[q4]);
      tc::tmem_wait_ld();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[B_SFREE + b]);

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
      const float nbias = (m_run == -INFINITY) ? 0.f : -m_run;
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};
      // P in place: pair i of column block q4 goes to word 16 q4 + i
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
      // the previous P.V must be done before P and O are touched
      if (j >= 1) ok = __all_sync(0xffffffffu, tt::wait_bar(c, B_ODONE, (j - 1) & 1));
      if (!ok) break;
      tc::tc_fence_after();
      tc::tmem_st32(lt + T_P, s[0]);
      tc::tmem_st32(lt + T_P + 32, s[1]);
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int q8 = 0; q8 < 4; ++q8) {
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
    }
    // ---- epilogue ----
    if (ok) ok = __all_sync(0xffffffffu, tt::wait_bar(c, B_FINAL, 0));
    tc::tc_fence_after();
    if (ok) {
      const bool st = valid && l_run > 0.f;
      const float inv = st ? 1.f / l_run : 0.f;
      uint16_t* dst = st ? a.out + (row * a.Hq + head) * DH : nullptr;
#pragma unroll 1
      for (int q8 = 0; q8 < 4; ++q8) {
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

}  // namespace sp
}  // namespace rk

struct rk_segpaged_plan_s {
  int device = -1;
  bool host_only = false;
  int32_t Hq = 0, Hkv = 0, G = 0, sink = 0, window = 0, max_blocks = 0;
  float scale = 0.f;
  int64_t num_pages = 0, rows = 0;
  rk_segpaged_info_t info{};
  std::vector<rk::sp::Req> reqs;
  std::vector<rk::sp::Tile> tiles;
  std::vector<int32_t> table;
  std::vector<uint8_t> role;
  rk::sp::Req* d_reqs = nullptr;
  rk::sp::Tile* d_tiles = nullptr;
  int32_t* d_table = nullptr;
  uint8_t* d_role = nullptr;
  int32_t* d_status = nullptr;
};

namespace {

using rk::sp::PAGE;

void sp_free(rk_segpaged_plan_s* p) {
  cudaFree(p->d_reqs);
  cudaFree(p->d_tiles);
  cudaFree(p->d_table);
  cudaFree(p->d_role);
  cudaFree(p->d_status);
  p->d_reqs = nullptr;
  p->d_tiles = nullptr;
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
  const int RT = 128 / G;
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
  rk_segpaged_info_t& info = p->info;
  info = rk_segpaged_info_t{};
  info.group = G;
  std::vector<std::pair<int64_t, rk::sp::Tile>> list;
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
        info.performed_pairs += int64_t(nb) * 128 * PAGE;
        list.push_back({nb, t});
      }
    }
    rows += T - qb;
  }
  if (rows * d->num_q_heads > (int64_t(1) << 40) || list.size() > INT32_MAX / 2)
    return RK_ERR_CAPACITY;
  std::stable_sort(list.begin(), list.end(),
                   [](const auto& x, const auto& y) { return x.first > y.first; });
  for (auto& e : list) p->tiles.push_back(e.second);
  p->rows = rows;
  info.rows = rows;
  info.tiles = static_cast<int64_t>(p->tiles.size());
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
    if (st == RK_OK) st = sp_upload(p->table, &p->d_table, s);
    if (st == RK_OK) st = sp_upload(p->role, &p->d_role, s);
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
                                           void* stream) {
  if (!p || !q || !k_pages || !v_pages || !out || !lse) return RK_ERR_NULL;
  if (p->host_only) return RK_ERR_PLAN_MISMATCH;
  auto mis = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) != 0; };
  if (mis(q) || mis(k_pages) || mis(v_pages) || mis(out) || (reinterpret_cast<uintptr_t>(lse) & 3))
    return RK_ERR_ALIGNMENT;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return RK_ERR_CUDA;
  if (cur != p->device) return RK_ERR_PLAN_MISMATCH;
  if (p->tiles.empty()) return RK_OK;
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
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaFuncSetAttribute(rk::sp::seg_paged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(rk::sp::SMEM_BYTES)) != cudaSuccess)
    return RK_ERR_CUDA;
  rk::sp::seg_paged_kernel<<<static_cast<unsigned>(p->tiles.size()), rk::sp::THREADS,
                             rk::sp::SMEM_BYTES, s>>>(a, mp);
  return cudaGetLastError() == cudaSuccess ? RK_OK : RK_ERR_CUDA;
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
