// Split-over-segments attention for single-row (decode) requests, Global
// heads, with a fused log-sum-exp merge.
//
// Each CTA takes one chunk: up to a few thousand keys of ONE segment of one
// request, for a group of 8 Global heads.  It rotates the 8 query RoPE
// slices by the segment's -delta once (RedKnot-MLA paper, RoPE-orthogonality
// paragraph), streams the canonical latent rows through shared memory, and
// keeps a running (max, sum, output) per head.  The chunk's normalised
// partial output and LSE go to the workspace; the last CTA of the request
// (atomic ticket) merges all partials with a numerically stable
// log-sum-exp and writes bf16 output and fp32 LSE.
//
// The contraction is laid out transposed: keys and d_v rows are the 16-row
// side of the mma.sync tile and the 8 heads are the 8-column side, so no
// tile padding is wasted on 8 heads.  The work is bound by HBM reads of the
// latent; the tensor path only keeps arithmetic off the critical path.

#include "common.cuh"
#include "tc_ptx.cuh"

namespace rk {
namespace {

constexpr int THREADS = 128;
constexpr int TK = 64;        // keys per shared-memory tile (16 per warp)
constexpr int NH = 8;         // heads per chunk

template <int DN, int DR, bool VROPE>
struct SCfg {
  static constexpr int DK = DN + DR;
  static constexpr int DV = VROPE ? DK : DN;  // V = c_nope, or the whole latent row
  static constexpr int QS = DN + 2 * DR + 8;
  static constexpr int KS = DK + 8;
  static constexpr int PS = TK + 8;
  static constexpr int DVW = DV / 4;       // d_v rows per warp
  static constexpr int MT = DVW / 16;      // output m-tiles per warp
  static constexpr int KSTEPS = (DN + 2 * DR) / 16;
  static constexpr size_t Q_BYTES = size_t(NH) * QS * 2;
  static constexpr size_t QRO_BYTES = size_t(NH) * DR * 2;
  static constexpr size_t K_BYTES = size_t(TK) * KS * 2;
  static constexpr size_t P_BYTES = size_t(NH) * PS * 2;
  static constexpr size_t SMEM = Q_BYTES + QRO_BYTES + 2 * K_BYTES + P_BYTES + 2 * 4 * NH * 4 + 16;
};

template <int DN, int DR, bool VROPE>
__global__ void __launch_bounds__(THREADS, 1) split_decode_kernel(const KernelArgs a) {
  using C = SCfg<DN, DR, VROPE>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Qro = reinterpret_cast<uint16_t*>(smem + C::Q_BYTES);
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem + C::Q_BYTES + C::QRO_BYTES);
  uint16_t* Ps = reinterpret_cast<uint16_t*>(smem + C::Q_BYTES + C::QRO_BYTES + 2 * C::K_BYTES);
  float* red_m = reinterpret_cast<float*>(smem + C::Q_BYTES + C::QRO_BYTES + 2 * C::K_BYTES +
                                          C::P_BYTES);
  float* red_l = red_m + 4 * NH;
  int* flag = reinterpret_cast<int*>(red_l + 4 * NH);

  const SplitChunk ch = a.chunks[blockIdx.x];
  const DevReq rq = a.reqs[ch.req];
  const DevSeg sg = a.segs[ch.seg];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int hbase = ch.group * NH;
  const int nh = min(NH, a.num_global - hbase);
  const int64_t frow = rq.row_base;  // the request's single computed row

  // ---- query rows of the 8 heads ----
  {
    constexpr int CH_N = DN / 8, CH_R = DR / 8, CH = CH_N + CH_R;
    for (int idx = tid; idx < NH * CH; idx += THREADS) {
      const int h = idx / CH, c = idx - h * CH;
      const uint16_t* src = a.q;
      int bytes = 0;
      if (h < nh) {
        src = a.q + (frow * a.H + a.global_heads[hbase + h]) * C::DK + c * 8;
        bytes = 16;
      }
      const uint32_t dst = (c < CH_N) ? smem_u32(Qs + h * C::QS + c * 8)
                                      : smem_u32(Qro + h * DR + (c - CH_N) * 8);
      cp_async16(dst, src, bytes);
    }
    cp_async_commit();
  }
  auto load_keys = [&](int k0, int stage) {
    constexpr int CH = C::DK / 8;
    uint16_t* dstb = Ks + stage * (TK * C::KS);
    for (int idx = tid; idx < TK * CH; idx += THREADS) {
      const int r = idx / CH, c = idx - r * CH;
      const int key = k0 + r;
      const bool ok = key < ch.k1;
      const uint16_t* src = ok ? sg.latent + int64_t(key - sg.delta) * C::DK + c * 8 : sg.latent;
      cp_async16(smem_u32(dstb + r * C::KS + c * 8), src, ok ? 16 : 0);
    }
  };
  load_keys(ch.k0, 0);
  cp_async_commit();
  cp_async_wait<1>();
  __syncthreads();
  // rotate q_rope by -delta (hi + lo bf16 parts)
  {
    const float* cs = a.rope_cs + int64_t(ch.seg) * DR;
    for (int idx = tid; idx < NH * (DR / 2); idx += THREADS) {
      const int h = idx / (DR / 2), j = idx - h * (DR / 2);
      const float c = cs[2 * j], s = cs[2 * j + 1];
      const uint32_t xy = *reinterpret_cast<const uint32_t*>(Qro + h * DR + 2 * j);
      const float x = __uint_as_float(xy << 16), y = __uint_as_float(xy & 0xffff0000u);
      const float xr = fmaf(x, c, y * s);
      const float yr = fmaf(-x, s, y * c);
      const uint32_t hi = pack_bf16x2(xr, yr);
      const float xh = __uint_as_float(hi << 16), yh = __uint_as_float(hi & 0xffff0000u);
      *reinterpret_cast<uint32_t*>(Qs + h * C::QS + DN + 2 * j) = hi;
      *reinterpret_cast<uint32_t*>(Qs + h * C::QS + DN + DR + 2 * j) = pack_bf16x2(xr - xh, yr - yh);
    }
  }
  __syncthreads();
  // Q^T as mma B fragments (k = dims, n = heads), kept in registers
  uint32_t qb[C::KSTEPS][2];
  {
    const uint32_t base = smem_u32(Qs + (lane & 7) * C::QS + 8 * (lane >> 3));
#pragma unroll
    for (int kk = 0; kk < C::KSTEPS / 2; ++kk) {
      uint32_t r[4];
      ldsm_x4(r, base + kk * 64);
      qb[2 * kk][0] = r[0];
      qb[2 * kk][1] = r[1];
      qb[2 * kk + 1][0] = r[2];
      qb[2 * kk + 1][1] = r[3];
    }
  }

  float o[C::MT][4];
#pragma unroll
  for (int i = 0; i < C::MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrun[2] = {-INFINITY, -INFINITY};  // heads 2*t4, 2*t4+1
  float lrun[2] = {0.f, 0.f};              // this warp's share of the sum
  const float sl2 = a.scale_log2;
  int stage = 0;
  for (int k0 = ch.k0; k0 < ch.k1; k0 += TK) {
    const bool more = k0 + TK < ch.k1;
    if (more) load_keys(k0 + TK, stage ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint16_t* Kt = Ks + stage * (TK * C::KS);
    // S^T: 16 keys of this warp x 8 heads
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t ka = smem_u32(Kt + (warp * 16 + (lane & 15)) * C::KS + 8 * (lane >> 4));
#pragma unroll
    for (int kk = 0; kk < DN / 16; ++kk) {
      uint32_t af[4];
      ldsm_x4(af, ka + kk * 32);
      mma16816(s, af, qb[kk][0], qb[kk][1]);
    }
#pragma unroll
    for (int kk = 0; kk < DR / 16; ++kk) {
      uint32_t af[4];
      ldsm_x4(af, ka + (DN + kk * 16) * 2);
      mma16816(s, af, qb[DN / 16 + kk][0], qb[DN / 16 + kk][1]);
      mma16816(s, af, qb[DN / 16 + DR / 16 + kk][0], qb[DN / 16 + DR / 16 + kk][1]);
    }
    const int key0 = k0 + warp * 16 + g;
    const bool v0 = key0 < ch.k1, v1 = key0 + 8 < ch.k1;
    s[0] = v0 ? s[0] * sl2 : -INFINITY;
    s[1] = v0 ? s[1] * sl2 : -INFINITY;
    s[2] = v1 ? s[2] * sl2 : -INFINITY;
    s[3] = v1 ? s[3] * sl2 : -INFINITY;
    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    if (g == 0) {
      red_m[warp * NH + 2 * t4] = mx0;
      red_m[warp * NH + 2 * t4 + 1] = mx1;
    }
    __syncthreads();
    float alpha[2], base[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float tm = red_m[2 * t4 + e];
#pragma unroll
      for (int w = 1; w < 4; ++w) tm = fmaxf(tm, red_m[w * NH + 2 * t4 + e]);
      const float mn = fmaxf(mrun[e], tm);
      if (mn == -INFINITY) {
        alpha[e] = 1.f;
        base[e] = 0.f;
      } else {
        alpha[e] = fast_exp2(mrun[e] - mn);
        base[e] = mn;
      }
      mrun[e] = mn;
    }
    const float p0 = fast_exp2(s[0] - base[0]), p1 = fast_exp2(s[1] - base[1]);
    const float p2 = fast_exp2(s[2] - base[0]), p3 = fast_exp2(s[3] - base[1]);
    const int kl = warp * 16 + g;
    Ps[(2 * t4) * C::PS + kl] = f32_to_bf16(p0);
    Ps[(2 * t4 + 1) * C::PS + kl] = f32_to_bf16(p1);
    Ps[(2 * t4) * C::PS + kl + 8] = f32_to_bf16(p2);
    Ps[(2 * t4 + 1) * C::PS + kl + 8] = f32_to_bf16(p3);
    float ls0 = p0 + p2, ls1 = p1 + p3;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, off);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, off);
    }
    lrun[0] = lrun[0] * alpha[0] + ls0;
    lrun[1] = lrun[1] * alpha[1] + ls1;
#pragma unroll
    for (int i = 0; i < C::MT; ++i) {
      o[i][0] *= alpha[0];
      o[i][1] *= alpha[1];
      o[i][2] *= alpha[0];
      o[i][3] *= alpha[1];
    }
    __syncthreads();
    // O^T[dims, heads] += V^T[dims, keys] P^T[keys, heads]
    uint32_t pb[4][2];
    {
      const uint32_t pbase = smem_u32(Ps + (lane & 7) * C::PS + 8 * (lane >> 3));
      uint32_t r[4];
      ldsm_x4(r, pbase);
      pb[0][0] = r[0]; pb[0][1] = r[1]; pb[1][0] = r[2]; pb[1][1] = r[3];
      ldsm_x4(r, pbase + 64);
      pb[2][0] = r[0]; pb[2][1] = r[1]; pb[3][0] = r[2]; pb[3][1] = r[3];
    }
    const uint32_t va = smem_u32(Kt + ((lane & 7) + 8 * (lane >> 4)) * C::KS + warp * C::DVW +
                                 8 * ((lane >> 3) & 1));
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt) {
        uint32_t af[4];
        ldsm_x4_t(af, va + (ks * 16 * C::KS + mt * 16) * 2);
        mma16816(o[mt], af, pb[ks][0], pb[ks][1]);
      }
    }
    __syncthreads();
    stage ^= 1;
  }
  cp_async_wait<0>();

  // ---- chunk partial: normalise by the sum over the 4 warps ----
  if (g == 0) {
    red_l[warp * NH + 2 * t4] = lrun[0];
    red_l[warp * NH + 2 * t4 + 1] = lrun[1];
  }
  __syncthreads();
  float lt[2];
#pragma unroll
  for (int e = 0; e < 2; ++e)
    lt[e] = red_l[2 * t4 + e] + red_l[NH + 2 * t4 + e] + red_l[2 * NH + 2 * t4 + e] +
            red_l[3 * NH + 2 * t4 + e];
  float* wo = a.ws_o + int64_t(ch.part) * NH * C::DV;
#pragma unroll
  for (int mt = 0; mt < C::MT; ++mt) {
    const int d0 = warp * C::DVW + mt * 16 + g;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = 2 * t4 + e;
      const float inv = 1.f / lt[e];
      wo[h * C::DV + d0] = o[mt][e] * inv;
      wo[h * C::DV + d0 + 8] = o[mt][2 + e] * inv;
    }
  }
  if (VROPE) {
    // the chunk lies in one segment: R(+delta) restores its output phase
    // before the merge (RedKnot-MLA paper, RoPE-orthogonality paragraph)
    __syncthreads();
    const float* cs = a.rope_cs + int64_t(ch.seg) * DR;
    for (int idx = tid; idx < NH * (DR / 2); idx += THREADS) {
      const int h = idx / (DR / 2), k = idx - h * (DR / 2);
      float* w2 = wo + h * C::DV + DN + 2 * k;
      const float c = cs[2 * k], sn = cs[2 * k + 1];
      const float x = w2[0], y = w2[1];
      w2[0] = x * c - y * sn;
      w2[1] = fmaf(x, sn, y * c);
    }
  }
  if (warp == 0 && g == 0) {
    a.ws_lse[int64_t(ch.part) * NH + 2 * t4] = mrun[0] * 0.6931471805599453f + logf(lt[0]);
    a.ws_lse[int64_t(ch.part) * NH + 2 * t4 + 1] = mrun[1] * 0.6931471805599453f + logf(lt[1]);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) flag[0] = (atomicAdd(a.ws_ticket + ch.mgroup, 1) == ch.nparts - 1);
  __syncthreads();
  if (!flag[0]) return;
  __threadfence();

  // ---- last CTA of the request: log-sum-exp merge of all partials ----
  for (int h = 0; h < nh; ++h) {
    float m = -INFINITY;
    for (int j = 0; j < ch.nparts; ++j)
      m = fmaxf(m, __ldcg(a.ws_lse + int64_t(ch.part_first + j) * NH + h));
    float ssum = 0.f;
    for (int j = 0; j < ch.nparts; ++j)
      ssum += __expf(__ldcg(a.ws_lse + int64_t(ch.part_first + j) * NH + h) - m);
    const int head = a.global_heads[hbase + h];
    uint16_t* dst = a.out + (frow * a.H + head) * C::DV;
    for (int d = 2 * tid; d < C::DV; d += 2 * THREADS) {
      float acc0 = 0.f, acc1 = 0.f;
      for (int j = 0; j < ch.nparts; ++j) {
        const int64_t pj = ch.part_first + j;
        const float w = __expf(__ldcg(a.ws_lse + pj * NH + h) - m);
        acc0 += w * __ldcg(a.ws_o + (pj * NH + h) * C::DV + d);
        acc1 += w * __ldcg(a.ws_o + (pj * NH + h) * C::DV + d + 1);
      }
      acc0 /= ssum;
      acc1 /= ssum;
      if (VROPE && d >= DN) {
        // inverse output RoPE R(-p) at the request's row p = 256 a + b
        const int k = (d - DN) >> 1, p = rq.q_row_begin;
        const float* hi = a.pos_cs_hi + int64_t(p >> 8) * DR + 2 * k;
        const float* lo = a.pos_cs_lo + int64_t(p & 255) * DR + 2 * k;
        const float pc = fmaf(hi[0], lo[0], -hi[1] * lo[1]);
        const float ps = fmaf(hi[1], lo[0], hi[0] * lo[1]);
        const float x = acc0, y = acc1;
        acc0 = fmaf(x, pc, y * ps);
        acc1 = fmaf(-x, ps, y * pc);
      }
      dst[d] = f32_to_bf16(acc0);
      dst[d + 1] = f32_to_bf16(acc1);
    }
    if (tid == 0) a.lse[frow * a.H + head] = m + logf(ssum);
  }
}


// ---------------------------------------------------------------------------
// Version fed by TMA for latent rows of NCH nope chunks + one rope chunk of
// 64 dims (d = 512 + 64, or 448 + 64 with the rotary value): each stage is
// one 3-D box of 32 keys x (NCH + 1) chunks (whole latent rows, laid out
// chunk-major with the 128-byte swizzle), five stages deep, so that four
// stages stay in flight while one is computed; fragment addresses apply the
// same XOR swizzle, so the ldmatrix reads are conflict-free.  Eight warps:
// the scores of the 32 keys are split over two key halves x four quarters
// of the 4 NCH + 8 k-steps (nope, then q_rope' hi and lo), each warp holding
// only its quarter of Q^T in registers, and each warp takes 64 of the 512
// output rows of P.V (V = the first 8 chunks: c_nope, or the whole row).
constexpr int DT_TK = 32;
constexpr int DT_ST = 5;                       // stages per CTA
constexpr int DT_THREADS = 256;
constexpr uint32_t DT_CH = DT_TK * 128;        // one 64-dim chunk of a stage
constexpr uint64_t DT_WAIT_NS = 2000000000ull;
constexpr int DT_PS = DT_TK + 8;
constexpr int DT_DV = 512;

template <int NCH>
struct TCfg {
  static constexpr int DN = 64 * NCH;
  static constexpr int DK = DN + 64;
  static constexpr int NKQ = NCH + 2;             // k-steps per quarter of d_k (+ rope lo)
  static constexpr uint32_t STAGE = (NCH + 1) * DT_CH;
  static constexpr int QS = DN + 128 + 8;         // [nope | rope hi | rope lo] + padding
  // shared-memory layout (byte offsets from the 1024-aligned base)
  static constexpr size_t OFF_Q = size_t(DT_ST) * STAGE;
  static constexpr size_t OFF_QRO = OFF_Q + size_t(NH) * QS * 2;
  static constexpr size_t OFF_P = OFF_QRO + size_t(NH) * 64 * 2;
  static constexpr size_t OFF_RED = OFF_P + size_t(NH) * DT_PS * 2;  // red_m [2][NH], red_l [2][NH]
  static constexpr size_t OFF_FLAG = OFF_RED + size_t(4) * NH * 4;
  static constexpr size_t OFF_BAR = (OFF_FLAG + 16 + 7) & ~size_t(7);
  static constexpr size_t OFF_PART = (OFF_BAR + size_t(DT_ST) * 8 + 15) & ~size_t(15);
  static constexpr size_t PART_BYTES = size_t(2) * 3 * 32 * 16;  // [key half][quarter 1..3][lane] float4
  static constexpr size_t SMEM = 1024 + OFF_PART + PART_BYTES;
  static_assert(OFF_Q % 16 == 0 && OFF_QRO % 16 == 0 && OFF_P % 16 == 0,
                "cp.async / ldmatrix targets are 16-byte aligned");
  static_assert(OFF_PART % 16 == 0 && OFF_BAR % 8 == 0, "float4 and mbarrier alignment");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(NCH >= 7 && NCH <= 8, "the last quarter holds 1 or 2 nope k-steps");
};

template <int NCH, bool VROPE>
__global__ void __launch_bounds__(DT_THREADS, 1) split_decode_tma_kernel(const KernelArgs a) {
  using T = TCfg<NCH>;
  constexpr uint32_t DT_STAGE = T::STAGE;
  constexpr int DT_QS = T::QS;
  constexpr size_t DT_OFF_Q = T::OFF_Q, DT_OFF_QRO = T::OFF_QRO, DT_OFF_P = T::OFF_P,
                   DT_OFF_RED = T::OFF_RED, DT_OFF_FLAG = T::OFF_FLAG, DT_OFF_BAR = T::OFF_BAR,
                   DT_OFF_PART = T::OFF_PART;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* Kst = sm;
  uint16_t* Qs = reinterpret_cast<uint16_t*>(sm + DT_OFF_Q);
  uint16_t* Qro = reinterpret_cast<uint16_t*>(sm + DT_OFF_QRO);
  uint16_t* Ps = reinterpret_cast<uint16_t*>(sm + DT_OFF_P);
  float* red_m = reinterpret_cast<float*>(sm + DT_OFF_RED);
  float* red_l = red_m + 2 * NH;
  int* flag = reinterpret_cast<int*>(sm + DT_OFF_FLAG);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + DT_OFF_BAR);
  float* part = reinterpret_cast<float*>(sm + DT_OFF_PART);

  const SplitChunk ch = a.chunks[blockIdx.x];
  const DevReq rq = a.reqs[ch.req];
  const DevSeg sg = a.segs[ch.seg];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int kq = warp >> 2, dq = warp & 3;  // key half, quarter of d_k
  const int hbase = ch.group * NH;
  const int nh = min(NH, a.num_global - hbase);
  const int64_t frow = rq.row_base;
  const int ntiles = (ch.k1 - ch.k0 + DT_TK - 1) / DT_TK;
  const CUtensorMap* map = a.decmaps + ch.seg;

  if (tid == 0) {
    for (int s = 0; s < DT_ST; ++s) tc::mbar_init(&full[s], 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    tc::prefetch_tmap(map);
    for (int s = 0; s < DT_ST && s < ntiles; ++s) {
      tc::mbar_arrive_expect_tx(&full[s], DT_STAGE);
      tc::tma_load_3d(smem_u32(Kst + s * DT_STAGE), map, &full[s], 0,
                      ch.k0 - sg.delta + s * DT_TK, 0);
    }
  }
  // ---- query rows of the 8 heads ----
  {
    constexpr int CH_N = T::DN / 8, CH = CH_N + 8;
    for (int idx = tid; idx < NH * CH; idx += DT_THREADS) {
      const int h = idx / CH, c = idx - h * CH;
      const uint16_t* src = a.q;
      int bytes = 0;
      if (h < nh) {
        src = a.q + (frow * a.H + a.global_heads[hbase + h]) * T::DK + c * 8;
        bytes = 16;
      }
      const uint32_t dst = (c < CH_N) ? smem_u32(Qs + h * DT_QS + c * 8)
                                      : smem_u32(Qro + h * 64 + (c - CH_N) * 8);
      cp_async16(dst, src, bytes);
    }
    cp_async_commit();
    cp_async_wait<0>();
  }
  __syncthreads();
  {
    const float* cs = a.rope_cs + int64_t(ch.seg) * 64;
    for (int idx = tid; idx < NH * 32; idx += DT_THREADS) {
      const int h = idx >> 5, j = idx & 31;
      const float c = cs[2 * j], s = cs[2 * j + 1];
      const uint32_t xy = *reinterpret_cast<const uint32_t*>(Qro + h * 64 + 2 * j);
      const float x = __uint_as_float(xy << 16), y = __uint_as_float(xy & 0xffff0000u);
      const float xr = fmaf(x, c, y * s), yr = fmaf(-x, s, y * c);
      const uint32_t hi = pack_bf16x2(xr, yr);
      const float xh = __uint_as_float(hi << 16), yh = __uint_as_float(hi & 0xffff0000u);
      *reinterpret_cast<uint32_t*>(Qs + h * DT_QS + T::DN + 2 * j) = hi;
      *reinterpret_cast<uint32_t*>(Qs + h * DT_QS + T::DN + 64 + 2 * j) =
          pack_bf16x2(xr - xh, yr - yh);
    }
  }
  __syncthreads();
  // this warp's NKQ k-steps of Q^T (k-steps NKQ dq .. NKQ dq + NKQ - 1 of
  // the 4 NKQ: nope, rope hi, rope lo) as mma B fragments; ten are loaded
  // (for NKQ = 9 the last one is not used)
  uint32_t qb[10][2];
  {
    const uint32_t base = smem_u32(Qs + (lane & 7) * DT_QS + 8 * (lane >> 3));
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      uint32_t r[4];
      ldsm_x4(r, base + (T::NKQ * dq + 2 * i) * 32);
      qb[2 * i][0] = r[0];
      qb[2 * i][1] = r[1];
      qb[2 * i + 1][0] = r[2];
      qb[2 * i + 1][1] = r[3];
    }
  }

  float o[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrun[2] = {-INFINITY, -INFINITY};
  float lrun[2] = {0.f, 0.f};
  const float sl2 = a.scale_log2;
  bool ok = true;
  int i = 0;
  for (; i < ntiles; ++i) {
    const int s = i % DT_ST;
    const bool got = tc::mbar_wait(&full[s], (i / DT_ST) & 1, a.status, DT_WAIT_NS);
    ok = __syncthreads_and(got) != 0;
    if (!ok) break;
    const uint32_t st = smem_u32(Kst + s * DT_STAGE);
    const int k0 = ch.k0 + i * DT_TK;
    // scores: warp (kq, dq) takes keys 16 kq.. over k-steps 10 dq.. on two
    // interleaved accumulators; the quarters are added through shared memory
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    {
      float sd[4] = {0.f, 0.f, 0.f, 0.f};
      const int r = kq * 16 + (lane & 15);
      const uint32_t rb = st + r * 128;
      const uint32_t rs = r & 7, hl = lane >> 4;
      // byte address of this lane's 16-byte row segment for k-step kk
      auto kaddr = [&](int kk) -> uint32_t {
        const uint32_t unit = ((static_cast<uint32_t>(kk) & 3u) << 1) | hl;
        return rb + static_cast<uint32_t>(kk >> 2) * DT_CH + ((unit ^ rs) << 4);
      };
      constexpr int NKQ = T::NKQ, NR = NCH - 6;  // nope k-steps of the last quarter
      if (dq < 3) {
#pragma unroll
        for (int j = 0; j < NKQ; j += 2) {
          uint32_t a0[4];
          ldsm_x4(a0, kaddr(NKQ * dq + j));
          mma16816(sc, a0, qb[j][0], qb[j][1]);
          if (j + 1 < NKQ) {
            uint32_t a1[4];
            ldsm_x4(a1, kaddr(NKQ * dq + j + 1));
            mma16816(sd, a1, qb[j + 1][0], qb[j + 1][1]);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < NR; ++i) {
          uint32_t a0[4];
          ldsm_x4(a0, kaddr(3 * NKQ + i));
          if (i & 1)
            mma16816(sd, a0, qb[i][0], qb[i][1]);
          else
            mma16816(sc, a0, qb[i][0], qb[i][1]);
        }
        // the rope chunk (k-steps 4 NCH ..) meets q_rope' hi and lo
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t af[4];
          ldsm_x4(af, kaddr(4 * NCH + kk));
          mma16816(sc, af, qb[NR + kk][0], qb[NR + kk][1]);
          mma16816(sd, af, qb[NR + 4 + kk][0], qb[NR + 4 + kk][1]);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[e] += sd[e];
      if (dq > 0)
        *reinterpret_cast<float4*>(part + ((kq * 3 + dq - 1) * 32 + lane) * 4) =
            make_float4(sc[0], sc[1], sc[2], sc[3]);
    }
    __syncthreads();
    if (dq == 0) {
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const float4 pt = *reinterpret_cast<const float4*>(part + ((kq * 3 + q) * 32 + lane) * 4);
        sc[0] += pt.x;
        sc[1] += pt.y;
        sc[2] += pt.z;
        sc[3] += pt.w;
      }
      const int key0 = k0 + kq * 16 + g;
      const bool v0 = key0 < ch.k1, v1 = key0 + 8 < ch.k1;
      sc[0] = v0 ? sc[0] * sl2 : -INFINITY;
      sc[1] = v0 ? sc[1] * sl2 : -INFINITY;
      sc[2] = v1 ? sc[2] * sl2 : -INFINITY;
      sc[3] = v1 ? sc[3] * sl2 : -INFINITY;
      float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      if (g == 0) {
        red_m[kq * NH + 2 * t4] = mx0;
        red_m[kq * NH + 2 * t4 + 1] = mx1;
      }
    }
    __syncthreads();
    float alpha[2], base[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float tm = fmaxf(red_m[2 * t4 + e], red_m[NH + 2 * t4 + e]);
      const float mn = fmaxf(mrun[e], tm);
      if (mn == -INFINITY) {
        alpha[e] = 1.f;
        base[e] = 0.f;
      } else {
        alpha[e] = fast_exp2(mrun[e] - mn);
        base[e] = mn;
      }
      mrun[e] = mn;
    }
    if (dq == 0) {
      const float p0 = fast_exp2(sc[0] - base[0]), p1 = fast_exp2(sc[1] - base[1]);
      const float p2 = fast_exp2(sc[2] - base[0]), p3 = fast_exp2(sc[3] - base[1]);
      const int kl = kq * 16 + g;
      Ps[(2 * t4) * DT_PS + kl] = f32_to_bf16(p0);
      Ps[(2 * t4 + 1) * DT_PS + kl] = f32_to_bf16(p1);
      Ps[(2 * t4) * DT_PS + kl + 8] = f32_to_bf16(p2);
      Ps[(2 * t4 + 1) * DT_PS + kl + 8] = f32_to_bf16(p3);
      float ls0 = p0 + p2, ls1 = p1 + p3;
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        ls0 += __shfl_xor_sync(0xffffffffu, ls0, off);
        ls1 += __shfl_xor_sync(0xffffffffu, ls1, off);
      }
      lrun[0] = lrun[0] * alpha[0] + ls0;
      lrun[1] = lrun[1] * alpha[1] + ls1;
    }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      o[mt][0] *= alpha[0];
      o[mt][1] *= alpha[1];
      o[mt][2] *= alpha[0];
      o[mt][3] *= alpha[1];
    }
    __syncthreads();
    // O^T[dims, heads] += V^T[dims, keys] P^T[keys, heads]; warp w: dims 64w..
    uint32_t pb[2][2];
    {
      uint32_t r[4];
      ldsm_x4(r, smem_u32(Ps + (lane & 7) * DT_PS + 8 * (lane >> 3)));
      pb[0][0] = r[0]; pb[0][1] = r[1]; pb[1][0] = r[2]; pb[1][1] = r[3];
    }
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const int key = 16 * ks + (lane & 7) + 8 * (lane >> 4);
      const uint32_t kb = st + key * 128;
      const uint32_t ks7 = key & 7;
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int dim = 64 * warp + 16 * mt + 8 * ((lane >> 3) & 1);
        uint32_t af[4];
        ldsm_x4_t(af, kb + (dim >> 6) * DT_CH + ((((dim & 63) >> 3) ^ ks7) << 4));
        mma16816(o[mt], af, pb[ks][0], pb[ks][1]);
      }
    }
    __syncthreads();
    if (tid == 0 && i + DT_ST < ntiles) {
      tc::mbar_arrive_expect_tx(&full[s], DT_STAGE);
      tc::tma_load_3d(st, map, &full[s], 0, ch.k0 - sg.delta + (i + DT_ST) * DT_TK, 0);
    }
  }
  if (!ok) {
    // drain the copies still in flight before the CTA exits
    if (tid == 0)
      for (int k = i; k < ntiles && k < i + DT_ST; ++k)
        tc::mbar_wait(&full[k % DT_ST], (k / DT_ST) & 1, a.status, DT_WAIT_NS);
    return;
  }

  // ---- chunk partial ----
  if (dq == 0 && g == 0) {
    red_l[kq * NH + 2 * t4] = lrun[0];
    red_l[kq * NH + 2 * t4 + 1] = lrun[1];
  }
  __syncthreads();
  float lt[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) lt[e] = red_l[2 * t4 + e] + red_l[NH + 2 * t4 + e];
  float* wo = a.ws_o + int64_t(ch.part) * NH * DT_DV;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
    const int d0 = 64 * warp + mt * 16 + g;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = 2 * t4 + e;
      const float inv = 1.f / lt[e];
      wo[h * DT_DV + d0] = o[mt][e] * inv;
      wo[h * DT_DV + d0 + 8] = o[mt][2 + e] * inv;
    }
  }
  if (VROPE) {
    // the chunk lies in one segment: R(+delta) restores its output phase
    // before the merge (RedKnot-MLA paper, RoPE-orthogonality paragraph)
    __syncthreads();
    const float* cs = a.rope_cs + int64_t(ch.seg) * 64;
    for (int idx = tid; idx < NH * 32; idx += DT_THREADS) {
      const int h = idx >> 5, k = idx & 31;
      float* w2 = wo + h * DT_DV + T::DN + 2 * k;
      const float c = cs[2 * k], sn = cs[2 * k + 1];
      const float x = w2[0], y = w2[1];
      w2[0] = x * c - y * sn;
      w2[1] = fmaf(x, sn, y * c);
    }
  }
  if (warp == 0 && g == 0) {
    a.ws_lse[int64_t(ch.part) * NH + 2 * t4] = mrun[0] * 0.6931471805599453f + logf(lt[0]);
    a.ws_lse[int64_t(ch.part) * NH + 2 * t4 + 1] = mrun[1] * 0.6931471805599453f + logf(lt[1]);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) flag[0] = (atomicAdd(a.ws_ticket + ch.mgroup, 1) == ch.nparts - 1);
  __syncthreads();
  if (!flag[0]) return;
  __threadfence();
  // ---- last CTA of the request: log-sum-exp merge of all partials ----
  // warp h finds head h's maximum and sum over the parts and writes each
  // part's weight exp(lse_j - m) / sum once into the idle stage ring (every
  // stage has landed and been consumed)
  const int np = ch.nparts;
  float* wts = reinterpret_cast<float*>(Kst);  // [NH][np]
  const bool in_smem = size_t(np) * NH * 4 <= size_t(DT_ST) * DT_STAGE;
  if (warp < nh) {
    const int h = warp;
    float m = -INFINITY;
    for (int j = lane; j < np; j += 32)
      m = fmaxf(m, __ldcg(a.ws_lse + int64_t(ch.part_first + j) * NH + h));
#pragma unroll
    for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float ssum = 0.f;
    for (int j = lane; j < np; j += 32)
      ssum += __expf(__ldcg(a.ws_lse + int64_t(ch.part_first + j) * NH + h) - m);
#pragma unroll
    for (int off = 16; off; off >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, off);
    if (in_smem)
      for (int j = lane; j < np; j += 32)
        wts[h * np + j] = __expf(__ldcg(a.ws_lse + int64_t(ch.part_first + j) * NH + h) - m) / ssum;
    if (lane == 0) {
      red_m[h] = m;
      red_l[h] = ssum;
    }
  }
  __syncthreads();
  for (int h = 0; h < nh; ++h) {
    const float m = red_m[h], ssum = red_l[h], inv = 1.f / ssum;
    const int head = a.global_heads[hbase + h];
    uint16_t* dst = a.out + (frow * a.H + head) * DT_DV;
    for (int d = 2 * tid; d < DT_DV; d += 2 * DT_THREADS) {
      float acc0 = 0.f, acc1 = 0.f;
      for (int j = 0; j < np; ++j) {
        const int64_t pj = ch.part_first + j;
        const float w = in_smem ? wts[h * np + j] : __expf(__ldcg(a.ws_lse + pj * NH + h) - m) * inv;
        const float2 x = __ldcg(reinterpret_cast<const float2*>(a.ws_o + (pj * NH + h) * DT_DV + d));
        acc0 = fmaf(w, x.x, acc0);
        acc1 = fmaf(w, x.y, acc1);
      }
      if (VROPE && d >= T::DN) {
        // inverse output RoPE R(-p) at the request's row p = 256 a + b
        const int k = (d - T::DN) >> 1, p = rq.q_row_begin;
        const float* hi = a.pos_cs_hi + int64_t(p >> 8) * 64 + 2 * k;
        const float* lo = a.pos_cs_lo + int64_t(p & 255) * 64 + 2 * k;
        const float pc = fmaf(hi[0], lo[0], -hi[1] * lo[1]);
        const float ps = fmaf(hi[1], lo[0], hi[0] * lo[1]);
        const float x = acc0, y = acc1;
        acc0 = fmaf(x, pc, y * ps);
        acc1 = fmaf(-x, ps, y * pc);
      }
      dst[d] = f32_to_bf16(acc0);
      dst[d + 1] = f32_to_bf16(acc1);
    }
    if (tid == 0) a.lse[frow * a.H + head] = m + logf(ssum);
  }
}

template <int DN, int DR, bool VROPE>
cudaError_t launch_t(const KernelArgs& a, cudaStream_t s) {
  using C = SCfg<DN, DR, VROPE>;
  auto k = split_decode_kernel<DN, DR, VROPE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  k<<<a.num_chunks, THREADS, C::SMEM, s>>>(a);
  return cudaGetLastError();
}

template <int NCH, bool VROPE>
cudaError_t launch_tma(const KernelArgs& a, cudaStream_t s) {
  auto k = split_decode_tma_kernel<NCH, VROPE>;
  constexpr size_t smem = TCfg<NCH>::SMEM;
  cudaError_t e =
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k<<<a.num_chunks, DT_THREADS, smem, s>>>(a);
  return cudaGetLastError();
}

// Stand-alone merge: one warp per (row, head) pair.
__global__ void lse_merge_kernel(const float* __restrict__ o_parts,
                                 const float* __restrict__ lse_parts, int P, int64_t pairs,
                                 int d_v, uint16_t* __restrict__ out, float* __restrict__ lse_out) {
  const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= pairs) return;
  float m = -INFINITY;
  for (int j = lane; j < P; j += 32) m = fmaxf(m, lse_parts[int64_t(j) * pairs + warp]);
#pragma unroll
  for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  uint16_t* dst = out + warp * d_v;
  if (m == -INFINITY) {
    for (int d = lane; d < d_v; d += 32) dst[d] = 0;
    if (lane == 0) lse_out[warp] = -INFINITY;
    return;
  }
  float ssum = 0.f;
  for (int j = lane; j < P; j += 32) ssum += __expf(lse_parts[int64_t(j) * pairs + warp] - m);
#pragma unroll
  for (int off = 16; off; off >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, off);
  const float inv = 1.f / ssum;
  for (int d = lane; d < d_v; d += 32) {
    float acc = 0.f;
    for (int j = 0; j < P; ++j) {
      const float l = lse_parts[int64_t(j) * pairs + warp];
      if (l == -INFINITY) continue;
      acc += __expf(l - m) * o_parts[(int64_t(j) * pairs + warp) * d_v + d];
    }
    dst[d] = f32_to_bf16(acc * inv);
  }
  if (lane == 0) lse_out[warp] = m + logf(ssum);
}

}  // namespace

cudaError_t launch_split_decode(const rk_seg_attn_plan_s& plan, const KernelArgs& a,
                                cudaStream_t s) {
  if (!plan.v_rope && plan.d_nope == 512 && plan.d_rope == 64 && a.decmaps)
    return launch_tma<8, false>(a, s);
  if (plan.v_rope && plan.d_nope == 448 && plan.d_rope == 64 && a.decmaps)
    return launch_tma<7, true>(a, s);
  if (plan.v_rope && plan.d_nope == 448 && plan.d_rope == 64) return launch_t<448, 64, true>(a, s);
  if (plan.d_nope == 512 && plan.d_rope == 64) return launch_t<512, 64, false>(a, s);
  if (plan.d_nope == 128 && plan.d_rope == 32) return launch_t<128, 32, false>(a, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int32_t P,
                             int64_t rows, int32_t H, int32_t d_v, uint16_t* out,
                             float* lse_out, cudaStream_t s) {
  const int64_t pairs = rows * H;
  const int64_t blocks = (pairs * 32 + 255) / 256;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  lse_merge_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(o_parts, lse_parts, P, pairs,
                                                                 d_v, out, lse_out);
  return cudaGetLastError();
}

}  // namespace rk
