// Projected state and layer output after the attention (RedKnot-MLA paper,
// first paragraphs: eqs. 2-4, the first output projection W_a sliced by the
// logical heads' channel ranges, y = W_b z; TP8 fast-path paragraph: sliced
// W_a projection, Local restoration and row-wise replacement into a
// contiguous projected state, W_b once; RedKnot blog, "The same idea on
// DeepSeek-V4": z = z_off + z_on).
//
// Heads act in their native output groups of 8; W_a holds one [d_g, 8 d_v]
// block per group.  For every computed row t and group g
//     z[t, g] = W_aG(g) O_G[t] + (row t protected ? W_aL(g) O_L[t] : z_off[t, g])
//     y[t]    = W_b z[t]
// (the inverse output rotation is the identity: the values carry no rotary
// part).  Two passes of one tcgen05 GEMM kernel on CTA pairs (M = 256 rows,
// 128 per CTA; N = 256 columns, 128 of the B rows loaded by each CTA;
// cta_group::2 MMAs issued by the first CTA; K in stages of two 64-wide
// chunks, one 32 KB box per operand and CTA, through a 3-stage ring):
//   pass z: A = the group's head outputs O[t, 8g + i, :], B = W_a rows; the
//           Global heads' chunks accumulate in tensor-memory columns 0..255,
//           the Local heads' chunks in 256..511, the latter only for row
//           tiles that hold a protected row; the epilogue adds z_off on the
//           unprotected rows instead and stores z (bf16).
//   pass y: A = z, B = W_b; the epilogue stores y (bf16).
// Every wait is bounded in time; on expiry the kernel records
// RK_ERR_DEVICE_TIMEOUT in the status word and stops.

#include "tc_tile.cuh"

namespace rk {
namespace {

using tt::Ctx;
using tt::drain_bar;
using tt::wait_bar;

constexpr int PJ_THREADS = 192;
constexpr int PJ_KC = 2;                   // 64-wide K chunks per stage (one box each)
constexpr uint32_t PJ_C = 16384;           // 128 rows x 64 bf16: one chunk of A or B
constexpr uint32_t PJ_A = PJ_KC * PJ_C;    // this CTA's rows
constexpr uint32_t PJ_B = PJ_KC * PJ_C;    // this CTA's half of N
constexpr uint32_t PJ_STAGE = PJ_A + PJ_B;
constexpr int PJ_ST = 3;
constexpr uint32_t PJ_OFF_BAR = PJ_ST * PJ_STAGE;
enum { P_FULL = 0, P_EMPTY = PJ_ST, P_DONE = 2 * PJ_ST, P_NBAR };
constexpr uint32_t PJ_SMEM = PJ_OFF_BAR + P_NBAR * 8 + 16 + 1024;
constexpr int PJ_MAX_GROUPS = 32;

struct ProjArgs {
  int32_t mode;            // 0: z pass, 1: y pass
  int64_t rows;
  int32_t groups;          // G
  int32_t dg;              // d_g
  int32_t dmodel;
  int32_t n_tiles;         // output columns / 256 (per group in pass z)
  const uint16_t* z_off;   // bf16 [rows, G, d_g]
  const uint32_t* prot;    // protected-row bits over the rows (LSB first)
  uint16_t* out;           // pass z: z bf16 [rows, G d_g]; pass y: y bf16 [rows, d_model]
  int32_t* status;
  uint8_t role_mask[PJ_MAX_GROUPS];  // bit i: head 8g + i is Global
};

// K-chunk c of the tile's walk -> (accumulator, chunk coordinate of A, of B).
// Pass z: the Global heads' 8 chunks each, then (if run) the Local heads'.
__device__ __forceinline__ void chunk_of(const ProjArgs& a, int g, int c, int& acc, int& ca,
                                         int& cb) {
  if (a.mode == 1) {
    acc = 0;
    ca = c;
    cb = c;
    return;
  }
  const uint32_t gm = a.role_mask[g];
  const int ng = __popc(gm);
  const bool local = c >= 8 * ng;
  const uint32_t set = local ? (~gm & 0xFFu) : gm;
  int k = local ? c - 8 * ng : c;
  int i = 0;
  for (; i < 8; ++i)  // the (k / 8)-th head of the set
    if ((set >> i) & 1u) {
      if (k < 8) break;
      k -= 8;
    }
  acc = local ? 1 : 0;
  ca = (8 * g + i) * 8 + k;   // O viewed as (64, rows, H * 8 chunks)
  cb = i * 8 + k;             // W_a viewed as (64, G d_g, 64 chunks)
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PJ_THREADS, 1)
    project_kernel(const __grid_constant__ ProjArgs a, const __grid_constant__ CUtensorMap ma,
                   const __grid_constant__ CUtensorMap mb) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + PJ_OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + PJ_OFF_BAR + P_NBAR * 8);
  const Ctx c{bar, reinterpret_cast<volatile uint32_t*>(misc + 1), a.status};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t r = tc::cluster_ctarank();  // this CTA's rows and half of the columns
  auto cbar = [&](int i, uint32_t rank) { return tc::mapa_shared(smem_u32(&bar[i]), rank); };
  // pair tile: (row tile of 256, group, column tile of 256) in pass z;
  // (row tile, column tile) in pass y
  const int pt = static_cast<int>(blockIdx.x >> 1);
  const int nt = pt % a.n_tiles;
  const int g = a.mode == 0 ? (pt / a.n_tiles) % a.groups : 0;
  const int64_t mt = a.mode == 0 ? pt / (a.n_tiles * a.groups) : pt / a.n_tiles;
  const int64_t mp = mt * 256;       // the pair's first row
  const int64_t m0 = mp + 128 * r;   // this CTA's first row
  // does the pair's row tile hold a protected row?  (pass z runs the Local
  // chunks only then; both CTAs take the same decision)
  bool any_prot = false;
  if (a.mode == 0) {
    for (int w = 0; w < 8; ++w) {
      const int64_t word = (mp >> 5) + w;
      if (word * 32 < a.rows && a.prot[word]) any_prot = true;
    }
  }
  const int ng = a.mode == 0 ? __popc(static_cast<uint32_t>(a.role_mask[g])) : 0;
  const int nchunks = a.mode == 0 ? 8 * ng + (any_prot ? 8 * (8 - ng) : 0) : a.dg / 64;
  const int32_t brow = (a.mode == 0 ? g * a.dg + nt * 256 : nt * 256) + 128 * static_cast<int32_t>(r);

  if (tid == 0) {
    for (int i = 0; i < PJ_ST; ++i) {
      tc::mbar_init(&bar[P_FULL + i], 1);
      tc::mbar_init(&bar[P_EMPTY + i], 1);
    }
    tc::mbar_init(&bar[P_DONE], 1);
    misc[1] = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc_2sm(misc, 512);
    tc::tmem_relinquish_2sm();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();  // both CTAs' barriers are initialised before any remote use
  tc::tc_fence_after();
  const uint32_t tbase = misc[0];

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      int k = 0;
      const int nst = nchunks / PJ_KC;
      for (; k < nst && ok; ++k) {
        const int s = k % PJ_ST;
        ok = wait_bar(c, P_EMPTY + s, ((k / PJ_ST) & 1) ^ 1);
        if (!ok) break;
        int acc, ca, cb;
        chunk_of(a, g, PJ_KC * k, acc, ca, cb);
        // the leader's barrier counts both CTAs' boxes
        if (r == 0) tc::mbar_arrive_expect_tx(&bar[P_FULL + s], 2 * PJ_STAGE);
        const uint32_t dst = smem_u32(sm + s * PJ_STAGE);
        tc::tma_load_3d_2sm(dst, &ma, cbar(P_FULL + s, 0), 0, static_cast<int32_t>(m0), ca);
        tc::tma_load_3d_2sm(dst + PJ_A, &mb, cbar(P_FULL + s, 0), 0, brow, cb);
      }
      // the pair's copies in flight land before either CTA may exit
      if (r == 0)
        for (int j = (k > PJ_ST ? k - PJ_ST : 0); j < k; ++j)
          drain_bar(c, P_FULL + j % PJ_ST, (j / PJ_ST) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && r == 0) {
      const uint32_t id = tc::idesc_bf16(256, 256, false, false);
      bool ok = true;
      bool first[2] = {true, true};
      const int nst = nchunks / PJ_KC;
      for (int k = 0; k < nst && ok; ++k) {
        const int s = k % PJ_ST;
        ok = wait_bar(c, P_FULL + s, (k / PJ_ST) & 1);
        if (!ok) break;
        tc::tc_fence_after();
        int acc, ca, cb;
        chunk_of(a, g, PJ_KC * k, acc, ca, cb);
        const uint32_t base = smem_u32(sm + s * PJ_STAGE);
#pragma unroll
        for (int kc = 0; kc < PJ_KC; ++kc)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            tc::mma_ss_2sm(tbase + 256 * acc, tc::sdesc_sw128(base + kc * PJ_C + 32 * kk, 16, 1024),
                           tc::sdesc_sw128(base + PJ_A + kc * PJ_C + 32 * kk, 16, 1024), id,
                           (first[acc] && kc == 0 && kk == 0) ? 0u : 1u);
          }
        first[acc] = false;
        tc::mma_commit_2sm(&bar[P_EMPTY + s], 0x3);
      }
      tc::mma_commit_2sm(&bar[P_DONE], 0x3);
    }
  } else {
    // ------------------------------------------------------ epilogue -----
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const int64_t row = m0 + m;
    const uint32_t lt = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const int ngc = a.mode == 0 ? __popc(static_cast<uint32_t>(a.role_mask[g])) : 1;
    const bool have_g = ngc > 0;
    const bool have_l = a.mode == 0 && any_prot && ngc < 8;
    const bool ok = __all_sync(0xffffffffu, wait_bar(c, P_DONE, 0));
    tc::tc_fence_after();
    if (ok) {
      const bool prot = a.mode == 0 && row < a.rows && ((a.prot[row >> 5] >> (row & 31)) & 1u);
      const int64_t ocols = a.mode == 0 ? int64_t(a.groups) * a.dg : a.dmodel;
      const int64_t ocol0 = a.mode == 0 ? int64_t(g) * a.dg + nt * 256 : int64_t(nt) * 256;
#pragma unroll 1
      for (int q = 0; q < 8; ++q) {
        uint32_t vg[32], vl[32];
        if (have_g) {
          tc::tmem_ld32(lt + 32 * q, vg);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) vg[i] = 0;
        }
        if (have_l) tc::tmem_ld32(lt + 256 + 32 * q, vl);
        tc::tmem_wait_ld();
        if (row >= a.rows) continue;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(vg[i]);
        if (a.mode == 0) {
          if (prot) {
            if (have_l) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] += __uint_as_float(vl[i]);
            }
          } else {
            // the cached projected Local contribution of this row
            const uint4* zo = reinterpret_cast<const uint4*>(
                a.z_off + row * ocols + ocol0 + 32 * q);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint4 w = __ldg(zo + u);
              const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                v[8 * u + 2 * e] += __uint_as_float(ww[e] << 16);
                v[8 * u + 2 * e + 1] += __uint_as_float(ww[e] & 0xffff0000u);
              }
            }
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(a.out + row * ocols + ocol0 + 32 * q);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4 w;
          w.x = pack_bf16x2(v[8 * u + 0], v[8 * u + 1]);
          w.y = pack_bf16x2(v[8 * u + 2], v[8 * u + 3]);
          w.z = pack_bf16x2(v[8 * u + 4], v[8 * u + 5]);
          w.w = pack_bf16x2(v[8 * u + 6], v[8 * u + 7]);
          dst[u] = w;
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) drain_bar(c, P_DONE, 0);  // the pair's MMA pipe is empty
  __syncthreads();
  tc::cluster_sync();  // no CTA leaves while the other may still use its memory
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc_2sm(tbase, 512);
  }
}

}  // namespace
}  // namespace rk

extern "C" rk_status_t rk_project_forward(const rk_project_desc_t* d, const void* o,
                                          const void* z_off, const uint32_t* prot,
                                          const void* w_a, const void* w_b, void* z, void* y,
                                          int32_t* status, void* stream) {
  using namespace rk;
  if (!d || !o || !z_off || !prot || !w_a || !w_b || !z || !y || !status || !d->head_role)
    return RK_ERR_NULL;
  if (d->rows < 1 || d->num_heads < 8 || d->num_heads % 8 || d->num_heads > 8 * PJ_MAX_GROUPS ||
      d->d_g < 256 || d->d_g % 256 || d->d_model < 256 || d->d_model % 256)
    return RK_ERR_INVALID_ARG;
  if (d->d_v != 512) return RK_ERR_UNSUPPORTED_DIMS;
  for (int h = 0; h < d->num_heads; ++h)
    if (d->head_role[h] > 1) return RK_ERR_INVALID_ARG;
  auto mis = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) != 0; };
  if (mis(o) || mis(z_off) || mis(w_a) || mis(w_b) || mis(z) || mis(y) ||
      (reinterpret_cast<uintptr_t>(prot) & 3) || (reinterpret_cast<uintptr_t>(status) & 3))
    return RK_ERR_ALIGNMENT;
  const int64_t rows = d->rows, H = d->num_heads, G = H / 8, dg = d->d_g, dm = d->d_model;
  if (rows > (int64_t(1) << 31) - 256) return RK_ERR_CAPACITY;
  const int64_t mtiles = (rows + 255) / 256;  // row tiles of a CTA pair
  if (2 * mtiles * G * (dg / 256) > INT32_MAX || 2 * mtiles * (dm / 256) > INT32_MAX)
    return RK_ERR_CAPACITY;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap ma{}, mb{};
  ProjArgs pa{};
  pa.rows = rows;
  pa.groups = static_cast<int32_t>(G);
  pa.dg = static_cast<int32_t>(dg);
  pa.dmodel = static_cast<int32_t>(dm);
  pa.z_off = static_cast<const uint16_t*>(z_off);
  pa.prot = prot;
  pa.status = status;
  for (int gg = 0; gg < G; ++gg) {
    uint8_t mk = 0;
    for (int i = 0; i < 8; ++i) mk |= (d->head_role[8 * gg + i] ? 1u : 0u) << i;
    pa.role_mask[gg] = mk;
  }
  if (cudaFuncSetAttribute(project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(PJ_SMEM)) != cudaSuccess)
    return RK_ERR_CUDA;
  // pass z: A = O viewed as (64, rows, H * 8 chunks); B = W_a as (64, G d_g, 64 chunks)
  {
    const uint64_t da[3] = {64, static_cast<uint64_t>(rows), static_cast<uint64_t>(H * 8)};
    const uint64_t sa[2] = {static_cast<uint64_t>(H) * 1024, 128};
    const uint32_t ba[3] = {64, 128, PJ_KC};
    const uint64_t db[3] = {64, static_cast<uint64_t>(G * dg), 64};
    const uint64_t sb[2] = {8 * 1024, 128};
    const uint32_t bb[3] = {64, 128, PJ_KC};
    if (!make_tmap_bf16(&ma, o, 3, da, sa, ba) || !make_tmap_bf16(&mb, w_a, 3, db, sb, bb))
      return RK_ERR_CUDA;
    pa.mode = 0;
    pa.n_tiles = static_cast<int32_t>(dg / 256);
    pa.out = static_cast<uint16_t*>(z);
    project_kernel<<<static_cast<unsigned>(2 * mtiles * G * (dg / 256)), PJ_THREADS, PJ_SMEM, s>>>(
        pa, ma, mb);
    if (cudaGetLastError() != cudaSuccess) return RK_ERR_CUDA;
  }
  // pass y: A = z as (64, rows, G d_g / 64 chunks); B = W_b as (64, d_model, G d_g / 64)
  {
    const uint64_t kc = static_cast<uint64_t>(G * dg / 64);
    const uint64_t da[3] = {64, static_cast<uint64_t>(rows), kc};
    const uint64_t sa[2] = {static_cast<uint64_t>(G * dg) * 2, 128};
    const uint32_t ba[3] = {64, 128, PJ_KC};
    const uint64_t db[3] = {64, static_cast<uint64_t>(dm), kc};
    const uint64_t sb[2] = {static_cast<uint64_t>(G * dg) * 2, 128};
    const uint32_t bb[3] = {64, 128, PJ_KC};
    if (!make_tmap_bf16(&ma, z, 3, da, sa, ba) || !make_tmap_bf16(&mb, w_b, 3, db, sb, bb))
      return RK_ERR_CUDA;
    pa.mode = 1;
    pa.dg = static_cast<int32_t>(G * dg);  // K of pass y
    pa.n_tiles = static_cast<int32_t>(dm / 256);
    pa.out = static_cast<uint16_t*>(y);
    project_kernel<<<static_cast<unsigned>(2 * mtiles * (dm / 256)), PJ_THREADS, PJ_SMEM, s>>>(
        pa, ma, mb);
    if (cudaGetLastError() != cudaSuccess) return RK_ERR_CUDA;
  }
  return RK_OK;
}
