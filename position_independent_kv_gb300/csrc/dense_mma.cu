// Prefill-style work tiles on the warp-level mma.sync tensor path.
//
// One CTA computes one tile of 64 (row, head) query pairs over the tile's
// key range, segment by segment: the query's RoPE slice is rotated by the
// segment's -delta (RedKnot-MLA paper, RoPE-orthogonality paragraph), scores
// are taken against the canonical latent rows in place (K = [c_nope |
// k_rope], V = c_nope of the same shared-memory rows), and one running
// online softmax per query carries across segments, which is the
// log-sum-exp merge of the per-segment statistics.  Global pairs see k <= p;
// Local pairs see the sink and [p - w, p] (RedKnot blog, "Insight 1").  The
// epilogue writes every pair of the tile; Local tiles only ever hold
// protected rows, so unprotected Local rows are never touched (paper,
// protected-set paragraph: replaced, never added).
//
// Warps 0-3 and 4-7 hold the two halves of d_v for the same 16 query pairs;
// both compute the same scores.  The rotated q_rope is kept as a bf16
// hi + lo pair so the rotation adds no rounding beyond fp32.

#include "common.cuh"

namespace rk {
namespace {

constexpr int TM = 64;
constexpr int TN = 32;
constexpr int THREADS = 256;

template <int DN, int DR>
struct Cfg {
  static constexpr int DK = DN + DR;
  static constexpr int QW = DN + 2 * DR;
  static constexpr int QS = QW + 8;     // q row stride (elements), 16-byte pad
  static constexpr int KS = DK + 8;     // key row stride (elements)
  static constexpr int DVH = DN / 2;    // d_v columns per warp
  static constexpr int NTO = DVH / 8;   // output n-tiles per warp
  static constexpr size_t Q_BYTES = size_t(TM) * QS * 2;
  static constexpr size_t QRO_BYTES = size_t(TM) * DR * 2;
  static constexpr size_t K_BYTES = size_t(TN) * KS * 2;
  static constexpr size_t SMEM = Q_BYTES + QRO_BYTES + 2 * K_BYTES;
};

template <int DN, int DR>
__global__ void __launch_bounds__(THREADS, 1) dense_mma_kernel(const KernelArgs a) {
  using C = Cfg<DN, DR>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Qro = reinterpret_cast<uint16_t*>(smem + C::Q_BYTES);
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem + C::Q_BYTES + C::QRO_BYTES);

  const DenseTile tile = a.tiles[blockIdx.x];
  const DevReq rq = a.reqs[tile.req];
  const DevSeg* segs = a.segs + rq.seg_first;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int mg = warp & 3, half = warp >> 2;
  const int g = lane >> 2, t4 = lane & 3;
  const bool is_global = tile.kind == 0;
  const int HG = a.num_global, HL = a.num_local;

  // (row, head) of query pair m; row < 0 marks an unused pair
  auto pair_of = [&](int m, int& row, int& head) {
    if (is_global) {
      const int r = m / HG;
      if (r < tile.count) {
        row = tile.first + r;
        head = a.global_heads[m - r * HG];
      } else {
        row = -1;
        head = 0;
      }
    } else {
      if (m < tile.count) {
        const int i = tile.first + m;
        const int lr = i / HL;
        row = a.local_rows[lr];
        head = a.local_heads[i - lr * HL];
      } else {
        row = -1;
        head = 0;
      }
    }
  };

  // ---- load the query tile (nope -> Qs, rope -> Qro) ----
  {
    constexpr int CH_N = DN / 8, CH_R = DR / 8, CH = CH_N + CH_R;
    for (int idx = tid; idx < TM * CH; idx += THREADS) {
      const int m = idx / CH, c = idx - m * CH;
      int row, head;
      pair_of(m, row, head);
      const uint16_t* src = a.q;
      int bytes = 0;
      if (row >= 0) {
        const int64_t fr = rq.row_base + (row - rq.q_row_begin);
        src = a.q + (fr * a.H + head) * C::DK + c * 8;
        bytes = 16;
      }
      const uint32_t dst = (c < CH_N) ? smem_u32(Qs + m * C::QS + c * 8)
                                      : smem_u32(Qro + m * DR + (c - CH_N) * 8);
      cp_async16(dst, src, bytes);
    }
    cp_async_commit();
  }

  // rows of this thread (g and g + 8 of the warp's 16) for masks/stores
  int prow[2], phead[2];
  pair_of(mg * 16 + g, prow[0], phead[0]);
  pair_of(mg * 16 + g + 8, prow[1], phead[1]);

  const int r0lo = 0, r0hi = tile.sink_hi, r1lo = tile.win_lo, r1hi = tile.key_hi;
  auto load_keys = [&](const KeyTile& kt, int stage) {
    const DevSeg sg = segs[kt.j];
    constexpr int CH = C::DK / 8;
    uint16_t* dstb = Ks + stage * (TN * C::KS);
    for (int idx = tid; idx < TN * CH; idx += THREADS) {
      const int r = idx / CH, c = idx - r * CH;
      const int key = kt.k0 + r;
      const bool ok = key < kt.k1;
      const uint16_t* src = ok ? sg.latent + int64_t(key - sg.delta) * C::DK + c * 8 : sg.latent;
      cp_async16(smem_u32(dstb + r * C::KS + c * 8), src, ok ? 16 : 0);
    }
  };

  KeyTile cur{0, 0, 0, -1};
  bool have = next_key_tile<TN>(cur, segs, rq.seg_count, r0lo, r0hi, r1lo, r1hi);
  KeyTile nxt = cur;
  bool have_next = have && next_key_tile<TN>(nxt, segs, rq.seg_count, r0lo, r0hi, r1lo, r1hi);
  if (have) load_keys(cur, 0);
  cp_async_commit();

  float o[C::NTO][4];
#pragma unroll
  for (int i = 0; i < C::NTO; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrun[2] = {-INFINITY, -INFINITY};
  float lrun[2] = {0.f, 0.f};
  int cur_seg = -1;
  int stage = 0;
  const float sl2 = a.scale_log2;
  const int sink = a.sink, window = a.window;

  while (have) {
    if (have_next) load_keys(nxt, stage ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (cur.j != cur_seg) {
      // rotate q_rope by -delta of this segment: hi + lo bf16 parts
      cur_seg = cur.j;
      const float* cs = a.rope_cs + int64_t(rq.seg_first + cur.j) * DR;
      for (int idx = tid; idx < TM * (DR / 2); idx += THREADS) {
        const int m = idx / (DR / 2), j = idx - m * (DR / 2);
        const float c = cs[2 * j], s = cs[2 * j + 1];
        const uint32_t xy = *reinterpret_cast<const uint32_t*>(Qro + m * DR + 2 * j);
        const float x = __uint_as_float(xy << 16), y = __uint_as_float(xy & 0xffff0000u);
        const float xr = fmaf(x, c, y * s);
        const float yr = fmaf(-x, s, y * c);
        const uint32_t hi = pack_bf16x2(xr, yr);
        const float xh = __uint_as_float(hi << 16), yh = __uint_as_float(hi & 0xffff0000u);
        const uint32_t lo = pack_bf16x2(xr - xh, yr - yh);
        *reinterpret_cast<uint32_t*>(Qs + m * C::QS + DN + 2 * j) = hi;
        *reinterpret_cast<uint32_t*>(Qs + m * C::QS + DN + DR + 2 * j) = lo;
      }
      __syncthreads();
    }
    const uint16_t* Kt = Ks + stage * (TN * C::KS);

    // ---- S = Q K^T for the warp's 16 pairs x 32 keys ----
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
    const uint32_t qa = smem_u32(Qs + (mg * 16 + (lane & 15)) * C::QS + (lane >> 4) * 8);
    const uint32_t kb0 =
        smem_u32(Kt + ((lane & 7) + 8 * (lane >> 4)) * C::KS + 8 * ((lane >> 3) & 1));
    const uint32_t kb1 = kb0 + 16 * C::KS * 2;
#pragma unroll 4
    for (int kk = 0; kk < DN / 16; ++kk) {
      uint32_t af[4], b0[4], b1[4];
      ldsm_x4(af, qa + kk * 32);
      ldsm_x4(b0, kb0 + kk * 32);
      ldsm_x4(b1, kb1 + kk * 32);
      mma16816(s[0], af, b0[0], b0[1]);
      mma16816(s[1], af, b0[2], b0[3]);
      mma16816(s[2], af, b1[0], b1[1]);
      mma16816(s[3], af, b1[2], b1[3]);
    }
#pragma unroll
    for (int kk = 0; kk < DR / 16; ++kk) {
      uint32_t ah[4], al[4], b0[4], b1[4];
      ldsm_x4(ah, qa + (DN + kk * 16) * 2);
      ldsm_x4(al, qa + (DN + DR + kk * 16) * 2);
      ldsm_x4(b0, kb0 + (DN + kk * 16) * 2);
      ldsm_x4(b1, kb1 + (DN + kk * 16) * 2);
      mma16816(s[0], ah, b0[0], b0[1]);
      mma16816(s[1], ah, b0[2], b0[3]);
      mma16816(s[2], ah, b1[0], b1[1]);
      mma16816(s[3], ah, b1[2], b1[3]);
      mma16816(s[0], al, b0[0], b0[1]);
      mma16816(s[1], al, b0[2], b0[3]);
      mma16816(s[2], al, b1[0], b1[1]);
      mma16816(s[3], al, b1[2], b1[3]);
    }

    // ---- masks + online softmax (log2 domain) ----
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = cur.k0 + nt * 8 + 2 * t4 + (e & 1);
        const int p = prow[e >> 1];
        bool vis = key < cur.k1 && key <= p;
        if (!is_global) vis = vis && (key < sink || key >= p - window);
        const float v = vis ? s[nt][e] * sl2 : -INFINITY;
        s[nt][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    }
    float alpha[2], base[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mn = fmaxf(mrun[r], mx[r]);
      if (mn == -INFINITY) {
        alpha[r] = 1.f;
        base[r] = 0.f;
      } else {
        alpha[r] = fast_exp2(mrun[r] - mn);
        base[r] = mn;
      }
      mrun[r] = mn;
    }
    float ls[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pv = fast_exp2(s[nt][e] - base[e >> 1]);
        s[nt][e] = pv;
        ls[e >> 1] += pv;
      }
    }
    lrun[0] = lrun[0] * alpha[0] + ls[0];
    lrun[1] = lrun[1] * alpha[1] + ls[1];
#pragma unroll
    for (int i = 0; i < C::NTO; ++i) {
      o[i][0] *= alpha[0];
      o[i][1] *= alpha[0];
      o[i][2] *= alpha[1];
      o[i][3] *= alpha[1];
    }

    // ---- O += P V over the warp's half of d_v ----
    const uint32_t vb = smem_u32(Kt + ((lane & 7) + 8 * ((lane >> 3) & 1)) * C::KS +
                                 half * C::DVH + 8 * (lane >> 4));
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(s[2 * ks][0], s[2 * ks][1]);
      pa[1] = pack_bf16x2(s[2 * ks][2], s[2 * ks][3]);
      pa[2] = pack_bf16x2(s[2 * ks + 1][0], s[2 * ks + 1][1]);
      pa[3] = pack_bf16x2(s[2 * ks + 1][2], s[2 * ks + 1][3]);
      const uint32_t vrow = vb + ks * 16 * C::KS * 2;
#pragma unroll
      for (int dp = 0; dp < C::NTO / 2; ++dp) {
        uint32_t b[4];
        ldsm_x4_t(b, vrow + dp * 32);
        mma16816(o[2 * dp], pa, b[0], b[1]);
        mma16816(o[2 * dp + 1], pa, b[2], b[3]);
      }
    }
    __syncthreads();
    cur = nxt;
    have = have_next;
    if (have) have_next = next_key_tile<TN>(nxt, segs, rq.seg_count, r0lo, r0hi, r1lo, r1hi);
    stage ^= 1;
  }
  cp_async_wait<0>();

  // ---- epilogue: normalise, LSE, store (replacement for Local pairs) ----
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float l = lrun[r];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    lrun[r] = l;
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (prow[r] < 0 || !(lrun[r] > 0.f)) continue;
    const float inv = 1.f / lrun[r];
    const int64_t fr = rq.row_base + (prow[r] - rq.q_row_begin);
    uint16_t* dst = a.out + (fr * a.H + phead[r]) * DN + half * C::DVH + 2 * t4;
#pragma unroll
    for (int nt = 0; nt < C::NTO; ++nt) {
      *reinterpret_cast<uint32_t*>(dst + nt * 8) =
          pack_bf16x2(o[nt][2 * r] * inv, o[nt][2 * r + 1] * inv);
    }
    if (half == 0 && t4 == 0)
      a.lse[fr * a.H + phead[r]] = mrun[r] * 0.6931471805599453f + logf(lrun[r]);
  }
}

template <int DN, int DR>
cudaError_t launch_t(const KernelArgs& a, cudaStream_t s) {
  using C = Cfg<DN, DR>;
  auto k = dense_mma_kernel<DN, DR>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  k<<<a.num_tiles, THREADS, C::SMEM, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dense_mma(const rk_seg_attn_plan_s& plan, const KernelArgs& a,
                             cudaStream_t s) {
  if (plan.d_nope == 512 && plan.d_rope == 64) return launch_t<512, 64>(a, s);
  if (plan.d_nope == 128 && plan.d_rope == 32) return launch_t<128, 32>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace rk
