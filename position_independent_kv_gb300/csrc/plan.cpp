// Host plan and C-ABI entry points of the segment-relocated MLA attention
// library.  The plan validates a request bundle, compacts the protected rows,
// builds the RoPE table and the work lists once; forward only launches.
// RedKnot-MLA paper (arXiv 2609.07008): TP8 fast-path paragraph (compact,
// reusable segment-pointer geometry), protected-set paragraph (which Local
// rows are recomputed), RoPE-orthogonality paragraph (query rotation by
// -delta and the log-sum-exp merge).

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <numeric>

#include "rk_internal.h"
#include "tmap.h"

using rk::DenseTile;
using rk::DevReq;
using rk::DevSeg;
using rk::SplitChunk;
using rk::TcPair;
using rk::TcTile;

namespace {

constexpr int kMmaTileM = 64;     // query pairs per mma.sync tile
constexpr int kMmaTileN = 32;     // keys per mma.sync key tile
constexpr int kSplitHeads = 8;    // Global heads per split chunk
constexpr int kTcM = 128;         // query pairs per tcgen05 tile
constexpr int kTcN = 128;         // keys per tcgen05 key tile

bool dims_supported(int d_nope, int d_rope, bool v_rope) {
  if (v_rope) return d_nope == 448 && d_rope == 64;
  return (d_nope == 512 && d_rope == 64) || (d_nope == 128 && d_rope == 32);
}

template <typename T>
rk_status_t upload(const std::vector<T>& v, T** dptr, cudaStream_t s) {
  *dptr = nullptr;
  if (v.empty()) return RK_OK;
  if (cudaMalloc(reinterpret_cast<void**>(dptr), v.size() * sizeof(T)) != cudaSuccess) {
    *dptr = nullptr;
    return RK_ERR_CUDA;
  }
  if (cudaMemcpyAsync(*dptr, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return RK_ERR_CUDA;
  return RK_OK;
}

void free_device(rk_seg_attn_plan_s* p) {
  cudaFree(p->d_segs);
  cudaFree(p->d_reqs);
  cudaFree(p->d_rope_cs);
  cudaFree(p->d_pos_cs_hi);
  cudaFree(p->d_pos_cs_lo);
  cudaFree(p->d_tiles);
  cudaFree(p->d_local_rows);
  cudaFree(p->d_global_heads);
  cudaFree(p->d_local_heads);
  cudaFree(p->d_chunks);
  cudaFree(p->d_tc_tiles);
  cudaFree(p->d_tc_pairs);
  cudaFree(p->d_tc_pairs_chunked);
  cudaFree(p->d_segmaps);
  cudaFree(p->d_decmaps);
  cudaFree(p->d_head_role);
  cudaFree(p->d_status);
  if (p->side) cudaStreamDestroy(p->side);
  if (p->ev_fork) cudaEventDestroy(p->ev_fork);
  if (p->ev_join) cudaEventDestroy(p->ev_join);
  p->side = nullptr;
  p->ev_fork = p->ev_join = nullptr;
  if (p->copy_in) cudaStreamDestroy(p->copy_in);
  if (p->copy_out) cudaStreamDestroy(p->copy_out);
  if (p->compute2) cudaStreamDestroy(p->compute2);
  for (cudaEvent_t* e : {&p->ev_start, &p->ev_split, &p->ev_done, &p->ev_c2})
    if (*e) cudaEventDestroy(*e);
  for (int c = 0; c < rk_seg_attn_plan_s::kHostChunks; ++c) {
    if (p->ev_in[c]) cudaEventDestroy(p->ev_in[c]);
    if (p->ev_k[c]) cudaEventDestroy(p->ev_k[c]);
    p->ev_in[c] = p->ev_k[c] = nullptr;
  }
  p->copy_in = p->copy_out = p->compute2 = nullptr;
  p->ev_start = p->ev_split = p->ev_done = p->ev_c2 = nullptr;
  p->d_tc_pairs_chunked = nullptr;
  p->d_segs = nullptr;
  p->d_reqs = nullptr;
  p->d_rope_cs = nullptr;
  p->d_pos_cs_hi = p->d_pos_cs_lo = nullptr;
  p->d_tiles = nullptr;
  p->d_local_rows = nullptr;
  p->d_global_heads = p->d_local_heads = nullptr;
  p->d_chunks = nullptr;
  p->d_tc_tiles = nullptr;
  p->d_tc_pairs = nullptr;
  p->d_segmaps = nullptr;
  p->d_decmaps = nullptr;
  p->d_head_role = nullptr;
  p->d_status = nullptr;
}

// Number of keys a tile visits in segment [d, d + n): the union
// [0, sink_hi) u [win_lo, key_hi) clipped to the segment, rounded up to key
// tiles of width `tn` per range.
int64_t key_tiles_in_segment(const DenseTile& t, int64_t d, int64_t n, int tn) {
  int64_t tiles = 0;
  auto add = [&](int64_t lo, int64_t hi) {
    lo = std::max(lo, d);
    hi = std::min(hi, d + n);
    if (hi > lo) tiles += (hi - lo + tn - 1) / tn;
  };
  add(0, t.sink_hi);
  add(t.win_lo, t.key_hi);
  return tiles;
}

int64_t keys_visible_local(int64_t p, int64_t sink, int64_t window) {
  int64_t lo = std::max<int64_t>(0, p - window);
  if (lo <= sink) return p + 1;
  return std::min<int64_t>(sink, p + 1) + (p - lo + 1);
}

}  // namespace

extern "C" const char* rk_status_string(rk_status_t s) {
  switch (s) {
    case RK_OK: return "ok";
    case RK_ERR_NULL: return "a required pointer is NULL";
    case RK_ERR_INVALID_ARG: return "invalid argument";
    case RK_ERR_SEGMENT_OVERLAP: return "segments of a request overlap";
    case RK_ERR_SEGMENT_GAP: return "segments of a request leave a gap";
    case RK_ERR_UNSUPPORTED_DIMS: return "unsupported (d_nope, d_rope)";
    case RK_ERR_CAPACITY: return "size exceeds a fixed limit";
    case RK_ERR_CUDA: return "CUDA call failed";
    case RK_ERR_DEVICE_TIMEOUT: return "bounded device-side wait expired";
    case RK_ERR_PLAN_MISMATCH: return "plan is host-only or belongs to another device";
    case RK_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case RK_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

static rk_status_t build_plan(const rk_seg_attn_desc_t* d, rk_seg_attn_plan_s* p) {
  // ---------------- validation (no CUDA call before this block ends) -----
  if (!d->seg_begin || !d->segs || !d->q_row_begin || !d->head_role) return RK_ERR_NULL;
  const int R = d->num_requests;
  if (R < 1) return RK_ERR_INVALID_ARG;
  if (d->num_heads < 8 || d->num_heads > 256 || d->num_heads % 8) return RK_ERR_INVALID_ARG;
  const bool v_rope = (d->flags & RK_PLAN_V_ROPE) != 0;
  if (!dims_supported(d->d_nope, d->d_rope, v_rope)) return RK_ERR_UNSUPPORTED_DIMS;
  if (!(d->rope_base > 1.0) || !std::isfinite(d->rope_base)) return RK_ERR_INVALID_ARG;
  if (!(d->softmax_scale > 0.f) || !std::isfinite(d->softmax_scale)) return RK_ERR_INVALID_ARG;
  if (d->sink < 0 || d->window < 0) return RK_ERR_INVALID_ARG;
  if (d->flags & ~(RK_PLAN_HOST_ONLY | RK_PLAN_LEGACY_MMA | RK_PLAN_SINGLE_CTA | RK_PLAN_CTA_PAIR |
                   RK_PLAN_NO_SIDE_PAIRS |
                   RK_PLAN_DEVICE_BITMAP | RK_PLAN_V_ROPE))
    return RK_ERR_INVALID_ARG;
  if (v_rope && (d->flags & (RK_PLAN_LEGACY_MMA | RK_PLAN_SINGLE_CTA | RK_PLAN_CTA_PAIR)))
    return RK_ERR_UNSUPPORTED_DIMS;
  if ((d->flags & RK_PLAN_DEVICE_BITMAP) && (d->flags & RK_PLAN_HOST_ONLY)) return RK_ERR_INVALID_ARG;
  if (d->seg_begin[0] != 0) return RK_ERR_INVALID_ARG;
  for (int r = 0; r < R; ++r)
    if (d->seg_begin[r + 1] <= d->seg_begin[r]) return RK_ERR_INVALID_ARG;
  const int64_t nseg = d->seg_begin[R];
  if (nseg > (1 << 24)) return RK_ERR_CAPACITY;
  const int H = d->num_heads;
  for (int h = 0; h < H; ++h)
    if (d->head_role[h] > 1) return RK_ERR_INVALID_ARG;
  for (int64_t i = 0; i < nseg; ++i) {
    const rk_segment_t& s = d->segs[i];
    if (!s.latent) return RK_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(s.latent) & 15) return RK_ERR_ALIGNMENT;
    if (s.n < 1 || s.delta < 0) return RK_ERR_INVALID_ARG;
    if ((s.flags & ~RK_SEG_NEW) || s.reserved) return RK_ERR_INVALID_ARG;
    if (s.n > INT32_MAX || s.delta > INT32_MAX) return RK_ERR_CAPACITY;
  }
  p->H = H;
  p->d_nope = d->d_nope;
  p->d_rope = d->d_rope;
  p->v_rope = v_rope;
  p->d_v = v_rope ? d->d_nope + d->d_rope : d->d_nope;
  p->sink = d->sink;
  p->window = d->window;
  p->softmax_scale = d->softmax_scale;
  p->host_only = (d->flags & RK_PLAN_HOST_ONLY) != 0;
  p->kernel = 0;
  p->tile_m = kMmaTileM;
  {
    int hg = 0;
    for (int h = 0; h < d->num_heads; ++h) hg += d->head_role[h] ? 1 : 0;
    const bool hg_ok = hg == 0 || (kTcM % hg == 0 && (kTcM / hg) % 8 == 0);
    const bool h_ok = d->num_heads == 64 || d->num_heads == 128;
    if (!(d->flags & RK_PLAN_LEGACY_MMA) && d->d_nope == 512 && d->d_rope == 64 && hg_ok && h_ok) {
      p->kernel = (d->flags & RK_PLAN_SINGLE_CTA) ? 1 : (d->flags & RK_PLAN_CTA_PAIR) ? 2 : 3;
      p->tile_m = kTcM;
    }
    // small heads (d_nope 128, d_rope 32): one tcgen05 CTA per tile of 128
    // query pairs of the generic work list
    if (!(d->flags & RK_PLAN_LEGACY_MMA) && !v_rope && d->d_nope == 128 && d->d_rope == 32 &&
        d->num_heads <= kTcM) {
      p->kernel = 4;
      p->tile_m = kTcM;
    }
    // the rotary value runs on the 4-CTA kernel only
    if (v_rope) {
      if (!(hg_ok && h_ok)) return RK_ERR_UNSUPPORTED_DIMS;
      p->kernel = 3;
      p->tile_m = kTcM;
    }
  }

  // segments, sorted by offset inside each request; contiguity check
  std::vector<int64_t> T(R), word_off(R + 1, 0);
  int64_t rows_total = 0;
  p->segs.resize(nseg);
  p->reqs.resize(R);
  for (int r = 0; r < R; ++r) {
    const int b = d->seg_begin[r], e = d->seg_begin[r + 1];
    std::vector<int> idx(e - b);
    std::iota(idx.begin(), idx.end(), b);
    std::stable_sort(idx.begin(), idx.end(),
                     [&](int x, int y) { return d->segs[x].delta < d->segs[y].delta; });
    int64_t pos = 0;
    for (int j = 0; j < e - b; ++j) {
      const rk_segment_t& s = d->segs[idx[j]];
      if (s.delta < pos) return RK_ERR_SEGMENT_OVERLAP;
      if (s.delta > pos) return RK_ERR_SEGMENT_GAP;
      pos = s.delta + s.n;
      if (pos > INT32_MAX) return RK_ERR_CAPACITY;
      DevSeg& ds = p->segs[b + j];
      ds.latent = static_cast<const uint16_t*>(s.latent);
      ds.n = static_cast<int32_t>(s.n);
      ds.delta = static_cast<int32_t>(s.delta);
      ds.is_new = (s.flags & RK_SEG_NEW) ? 1 : 0;
      ds.pad = 0;
    }
    T[r] = pos;
    const int64_t qb = d->q_row_begin[r];
    if (qb < 0 || qb >= pos) return RK_ERR_INVALID_ARG;
    DevReq& rq = p->reqs[r];
    rq.seg_first = b;
    rq.seg_count = e - b;
    rq.T = static_cast<int32_t>(pos);
    rq.q_row_begin = static_cast<int32_t>(qb);
    rq.row_base = rows_total;
    rows_total += pos - qb;
    word_off[r + 1] = word_off[r] + (pos + 31) / 32;
  }
  if (rows_total * H > (int64_t(1) << 40)) return RK_ERR_CAPACITY;
  // a device bitmap is brought to the host once the geometry is validated
  std::vector<uint32_t> host_bits;
  const uint32_t* bitmap = d->protected_bitmap;
  if (bitmap && (d->flags & RK_PLAN_DEVICE_BITMAP)) {
    host_bits.resize(static_cast<size_t>(word_off[R]));
    if (cudaMemcpy(host_bits.data(), bitmap, host_bits.size() * sizeof(uint32_t),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
      return RK_ERR_CUDA;
    bitmap = host_bits.data();
  }

  // heads
  for (int h = 0; h < H; ++h) (d->head_role[h] ? p->global_heads : p->local_heads).push_back(h);
  p->head_role.assign(d->head_role, d->head_role + H);
  if (static_cast<int>(p->global_heads.size()) == H / 8) {
    const int c0 = p->global_heads.empty() ? -1 : p->global_heads[0];
    bool pat = c0 >= 0 && c0 < 8;
    for (size_t g = 0; g < p->global_heads.size() && pat; ++g)
      pat = p->global_heads[g] == static_cast<int>(8 * g) + c0;
    p->g_ingroup = pat ? c0 : -1;
  }
  const int HG = static_cast<int>(p->global_heads.size());
  const int HL = static_cast<int>(p->local_heads.size());

  // RoPE table: cos/sin(delta * theta_j) in fp64, stored fp32
  const int half = d->d_rope / 2;
  p->rope_cs.resize(static_cast<size_t>(nseg) * half * 2);
  for (int64_t i = 0; i < nseg; ++i) {
    for (int j = 0; j < half; ++j) {
      const double theta = std::pow(d->rope_base, -2.0 * j / d->d_rope);
      const double ang = static_cast<double>(p->segs[i].delta) * theta;
      p->rope_cs[(i * half + j) * 2 + 0] = static_cast<float>(std::cos(ang));
      p->rope_cs[(i * half + j) * 2 + 1] = static_cast<float>(std::sin(ang));
    }
  }
  // inverse output RoPE at any query position p = 256 a + b: cos/sin(256 a
  // theta_j) and cos/sin(b theta_j), fp64 then fp32; the kernels combine the
  // two by the angle-addition formulas
  if (v_rope) {
    int64_t tmax = 0;
    for (int r = 0; r < R; ++r) tmax = std::max(tmax, T[r]);
    const int64_t nhi = tmax / 256 + 1;
    p->pos_cs_hi.resize(static_cast<size_t>(nhi) * half * 2);
    p->pos_cs_lo.resize(static_cast<size_t>(256) * half * 2);
    for (int j = 0; j < half; ++j) {
      const double theta = std::pow(d->rope_base, -2.0 * j / d->d_rope);
      for (int64_t a = 0; a < nhi; ++a) {
        const double ang = static_cast<double>(256 * a) * theta;
        p->pos_cs_hi[(a * half + j) * 2 + 0] = static_cast<float>(std::cos(ang));
        p->pos_cs_hi[(a * half + j) * 2 + 1] = static_cast<float>(std::sin(ang));
      }
      for (int64_t b = 0; b < 256; ++b) {
        const double ang = static_cast<double>(b) * theta;
        p->pos_cs_lo[(b * half + j) * 2 + 0] = static_cast<float>(std::cos(ang));
        p->pos_cs_lo[(b * half + j) * 2 + 1] = static_cast<float>(std::sin(ang));
      }
    }
  }

  // work lists
  rk_plan_info_t& info = p->info;
  std::memset(&info, 0, sizeof(info));
  info.rows = rows_total;
  info.num_heads = H;
  info.d_nope = d->d_nope;
  info.d_rope = d->d_rope;
  info.num_global_heads = HG;
  info.num_local_heads = HL;
  info.kernel = p->kernel;
  info.d_v = p->d_v;
  for (int64_t i = 0; i < nseg; ++i)
    info.latent_bytes += p->segs[i].n * int64_t(d->d_nope + d->d_rope) * 2;

  const int TM = p->tile_m;
  const bool tc = p->kernel >= 1 && p->kernel <= 3;  // tcgen05 tiles of the TcTile kind
  const int TN = (tc || p->kernel == 4) ? kTcN : kMmaTileN;
  const int64_t sink = d->sink, window = d->window;
  std::vector<std::pair<int64_t, DenseTile>> tiles;  // (cost, tile)
  std::vector<std::pair<int64_t, TcTile>> tc_list;   // (cost, tile)
  int64_t mgroups = 0, parts = 0;
  const int groups = (HG + kSplitHeads - 1) / kSplitHeads;
  for (int r = 0; r < R; ++r) {
    const DevReq& rq = p->reqs[r];
    const int64_t qb = rq.q_row_begin, Tr = rq.T;
    // protected computed rows
    std::vector<uint8_t> prot(Tr, 0);
    if (bitmap) {
      const uint32_t* w = bitmap + word_off[r];
      for (int64_t q = 0; q < Tr; ++q) prot[q] = (w[q >> 5] >> (q & 31)) & 1u;
    }
    for (int j = 0; j < rq.seg_count; ++j) {
      const DevSeg& s = p->segs[rq.seg_first + j];
      if (s.is_new) std::fill(prot.begin() + s.delta, prot.begin() + s.delta + s.n, 1);
    }
    const size_t lr_first = p->local_rows.size();
    for (int64_t q = qb; q < Tr; ++q)
      if (prot[q]) p->local_rows.push_back(static_cast<int32_t>(q));
    const int64_t nprot = static_cast<int64_t>(p->local_rows.size() - lr_first);
    if (HL) info.protected_local_rows += nprot;
    for (size_t i = lr_first; i < p->local_rows.size(); ++i) {
      const int64_t f = rq.row_base + (p->local_rows[i] - qb);
      if (!p->full_rows.empty() && p->full_rows.back().second == f)
        ++p->full_rows.back().second;
      else
        p->full_rows.push_back({f, f + 1});
    }

    // algorithmic pairs
    for (int64_t q = qb; q < Tr; ++q) info.pairs_global += int64_t(HG) * (q + 1);
    if (HL)
      for (size_t i = lr_first; i < p->local_rows.size(); ++i)
        info.pairs_local += int64_t(HL) * keys_visible_local(p->local_rows[i], sink, window);

    // Global heads
    const bool split = (Tr - qb == 1) && HG > 0;
    if (split) {
      // one row: split the keys [0, T) over segments and chunks
      const int64_t keys = Tr;
      int64_t C = (keys + 3) / 4;  // at least a few chunks per request
      C = std::max<int64_t>(256, std::min<int64_t>(4096, ((C + 63) / 64) * 64));
      for (int g = 0; g < groups; ++g) {
        const int64_t first = parts;
        std::vector<SplitChunk> cs;
        for (int j = 0; j < rq.seg_count; ++j) {
          const DevSeg& s = p->segs[rq.seg_first + j];
          for (int64_t k0 = s.delta; k0 < int64_t(s.delta) + s.n; k0 += C) {
            SplitChunk c{};
            c.req = r;
            c.seg = rq.seg_first + j;
            c.k0 = static_cast<int32_t>(k0);
            c.k1 = static_cast<int32_t>(std::min<int64_t>(k0 + C, int64_t(s.delta) + s.n));
            c.group = g;
            c.mgroup = static_cast<int32_t>(mgroups);
            cs.push_back(c);
          }
        }
        for (auto& c : cs) {
          c.part = static_cast<int32_t>(parts++);
          c.part_first = static_cast<int32_t>(first);
          c.nparts = static_cast<int32_t>(cs.size());
          p->chunks.push_back(c);
          info.performed_pairs += int64_t(kSplitHeads) * ((c.k1 - c.k0 + 63) / 64) * 64;
        }
        ++mgroups;
      }
    } else if (HG && tc) {
      const int rows_per = kTcM / HG;
      for (int64_t q0 = qb; q0 < Tr; q0 += rows_per) {
        TcTile t{};
        t.req = r;
        t.kind = 0;
        t.p0 = static_cast<int32_t>(q0);
        t.p1 = static_cast<int32_t>(std::min<int64_t>(rows_per, Tr - q0));
        t.key_hi = t.p0 + t.p1;
        DenseTile shape{};
        shape.key_hi = t.key_hi;
        int64_t kt = 0;
        for (int j = 0; j < rq.seg_count; ++j) {
          const DevSeg& s = p->segs[rq.seg_first + j];
          kt += key_tiles_in_segment(shape, s.delta, s.n, TN);
        }
        tc_list.push_back({kt, t});
      }
    } else if (HG) {
      const int rows_per = std::max(1, TM / HG);
      for (int64_t q0 = qb; q0 < Tr; q0 += rows_per) {
        DenseTile t{};
        t.req = r;
        t.kind = 0;
        t.first = static_cast<int32_t>(q0);
        t.count = static_cast<int32_t>(std::min<int64_t>(rows_per, Tr - q0));
        t.key_hi = t.first + t.count;
        t.win_lo = 0;
        t.sink_hi = 0;
        int64_t kt = 0;
        for (int j = 0; j < rq.seg_count; ++j) {
          const DevSeg& s = p->segs[rq.seg_first + j];
          kt += key_tiles_in_segment(t, s.delta, s.n, TN);
        }
        info.performed_pairs += kt * TN * TM;
        tiles.push_back({kt, t});
      }
    }
    // Local heads on protected rows.  A request whose only computed row is
    // its new row (decode) runs its Local heads as mma.sync tiles of 64
    // pairs x 32 keys: one row x the Local heads over at most w + 1 + sink
    // keys is too little work to fill a tcgen05 tile pair, whose partner
    // would be idle (tiles of two requests share no keys).  The rotary value
    // has no mma.sync form and keeps the 4-CTA tiles.
    const bool local_mma = tc && split && !v_rope;
    if (HL && nprot && tc && !local_mma) {
      const int rows_per = kTcM / H;  // 1 or 2 rows of every head per tile
      int64_t i = 0;
      while (i < nprot) {
        const int64_t pa = p->local_rows[lr_first + i];
        int64_t pb = -1;
        if (rows_per == 2 && i + 1 < nprot &&
            p->local_rows[lr_first + i + 1] - pa <= window / 2 + 1)
          pb = p->local_rows[lr_first + i + 1];
        TcTile t{};
        t.req = r;
        t.kind = 1;
        t.p0 = static_cast<int32_t>(pa);
        t.p1 = static_cast<int32_t>(pb);
        const int64_t plast = pb >= 0 ? pb : pa;
        t.key_hi = static_cast<int32_t>(plast + 1);
        const int64_t wl = std::max<int64_t>(0, pa - window);
        if (wl <= sink) {
          t.win_lo = 0;
          t.sink_hi = 0;
        } else {
          t.win_lo = static_cast<int32_t>(wl);
          t.sink_hi = static_cast<int32_t>(sink);
        }
        DenseTile shape{};
        shape.key_hi = t.key_hi;
        shape.win_lo = t.win_lo;
        shape.sink_hi = t.sink_hi;
        int64_t kt = 0;
        for (int j = 0; j < rq.seg_count; ++j) {
          const DevSeg& s = p->segs[rq.seg_first + j];
          kt += key_tiles_in_segment(shape, s.delta, s.n, TN);
        }
        tc_list.push_back({kt, t});
        i += pb >= 0 ? 2 : 1;
      }
    } else if (HL && nprot) {
      const int LTM = local_mma ? kMmaTileM : TM;
      const int LTN = local_mma ? kMmaTileN : TN;
      const int64_t npairs = nprot * HL;
      const int64_t pair_base = static_cast<int64_t>(lr_first) * HL;
      int64_t i = 0;
      while (i < npairs) {
        const int64_t p_first = p->local_rows[lr_first + i / HL];
        int64_t e = std::min<int64_t>(npairs, i + LTM);
        // cut the tile where the next row is too far away to share a window
        for (int64_t k = i + 1; k < e; ++k) {
          if ((k % HL) == 0 && p->local_rows[lr_first + k / HL] - p_first > window / 2 + 1) {
            e = k;
            break;
          }
        }
        const int64_t p_last = p->local_rows[lr_first + (e - 1) / HL];
        DenseTile t{};
        t.req = r;
        t.kind = 1;
        t.first = static_cast<int32_t>(pair_base + i);
        t.count = static_cast<int32_t>(e - i);
        t.key_hi = static_cast<int32_t>(p_last + 1);
        int64_t wl = std::max<int64_t>(0, p_first - window);
        if (wl <= sink) {
          t.win_lo = 0;
          t.sink_hi = 0;
        } else {
          t.win_lo = static_cast<int32_t>(wl);
          t.sink_hi = static_cast<int32_t>(sink);
        }
        int64_t kt = 0;
        for (int j = 0; j < rq.seg_count; ++j) {
          const DevSeg& s = p->segs[rq.seg_first + j];
          kt += key_tiles_in_segment(t, s.delta, s.n, LTN);
        }
        info.performed_pairs += kt * LTN * LTM;
        tiles.push_back({kt, t});
        i = e;
      }
    }
  }
  if (static_cast<int64_t>(p->local_rows.size()) * std::max(HL, 1) > INT32_MAX)
    return RK_ERR_CAPACITY;
  if (tiles.size() > INT32_MAX / 2 || p->chunks.size() > INT32_MAX / 2) return RK_ERR_CAPACITY;
  // longest chunks first (each chunk carries its own partial slot)
  std::stable_sort(p->chunks.begin(), p->chunks.end(), [](const SplitChunk& a, const SplitChunk& b) {
    return a.k1 - a.k0 > b.k1 - b.k0;
  });
  // longest first
  std::stable_sort(tiles.begin(), tiles.end(),
                   [](const auto& a, const auto& b) { return a.first > b.first; });
  p->tiles.reserve(tiles.size());
  for (auto& t : tiles) p->tiles.push_back(t.second);
  info.dense_tiles = static_cast<int64_t>(p->tiles.size() + tc_list.size());
  if (p->kernel >= 2) {
    // Pair neighbouring tiles of one request and kind (adjacent Global row
    // blocks, consecutive protected rows) when the union of their key
    // ranges costs at most 1/8 more key tiles than the two ranges apart;
    // a tile left alone gets a partner without work.
    auto req_tiles = [&](int r, int64_t sink_hi, int64_t win_lo, int64_t key_hi) {
      DenseTile shape{};
      shape.key_hi = static_cast<int32_t>(key_hi);
      shape.win_lo = static_cast<int32_t>(win_lo);
      shape.sink_hi = static_cast<int32_t>(sink_hi);
      int64_t kt = 0;
      const DevReq& rq = p->reqs[r];
      for (int j = 0; j < rq.seg_count; ++j) {
        const DevSeg& s = p->segs[rq.seg_first + j];
        kt += key_tiles_in_segment(shape, s.delta, s.n, TN);
      }
      return kt;
    };
    // segments of request `req` that meet neither [0, sh) nor [wl, ...):
    // those from the first one starting at or after sh up to the first one
    // ending after wl (segments are sorted by offset)
    auto skip_hint = [&](int req, int64_t sh, int64_t wl) -> int32_t {
      const DevReq& rq = p->reqs[req];
      if (wl <= sh || rq.seg_count > 0xffff) return 0;
      const DevSeg* sg = p->segs.data() + rq.seg_first;
      int lo = 0, hi = rq.seg_count;
      while (lo < hi) {  // first segment with delta >= sh
        const int mid = (lo + hi) / 2;
        if (sg[mid].delta < sh) lo = mid + 1; else hi = mid;
      }
      const int jlo = lo;
      hi = rq.seg_count;
      while (lo < hi) {  // first segment ending after wl
        const int mid = (lo + hi) / 2;
        if (int64_t(sg[mid].delta) + sg[mid].n <= wl) lo = mid + 1; else hi = mid;
      }
      return jlo < lo ? static_cast<int32_t>((static_cast<uint32_t>(lo) << 16) | uint32_t(jlo)) : 0;
    };
    std::vector<std::pair<int64_t, TcPair>> pairs;
    size_t i = 0;
    while (i < tc_list.size()) {
      const TcTile& A = tc_list[i].second;
      TcPair pr{};
      pr.t[0] = A;
      pr.key_hi = A.key_hi;
      pr.win_lo = A.win_lo;
      pr.sink_hi = A.sink_hi;
      int64_t cost = tc_list[i].first;
      bool paired = false;
      if (i + 1 < tc_list.size()) {
        const TcTile& B = tc_list[i + 1].second;
        if (B.req == A.req && B.kind == A.kind) {
          int64_t sh = std::max(A.sink_hi, B.sink_hi);
          int64_t wl = std::min(A.win_lo, B.win_lo);
          const int64_t kh = std::max(A.key_hi, B.key_hi);
          if (sh >= wl) sh = wl = 0;
          const int64_t u = req_tiles(A.req, sh, wl, kh);
          const int64_t apart = tc_list[i].first + tc_list[i + 1].first;
          if (2 * u <= apart + apart / 8) {
            pr.t[1] = B;
            pr.key_hi = static_cast<int32_t>(kh);
            pr.win_lo = static_cast<int32_t>(wl);
            pr.sink_hi = static_cast<int32_t>(sh);
            cost = u;
            paired = true;
          }
        }
      }
      if (!paired) {
        pr.t[1] = A;
        pr.t[1].pad |= 1;
      }
      pr.skip = skip_hint(A.req, pr.sink_hi, pr.win_lo);
      // both CTAs of a real pair do attention work; a partner without work does not count
      info.performed_pairs += (paired ? 2 : 1) * cost * TN * TM;
      pairs.push_back({cost, pr});
      i += paired ? 2 : 1;
    }
    std::stable_sort(pairs.begin(), pairs.end(),
                     [](const auto& a, const auto& b) { return a.first > b.first; });
    for (auto& pr : pairs) p->tc_pairs.push_back(pr.second);
    // the short tail that the side kernel beside the 4-CTA clusters may take
    p->side_pairs = 0;
    if (p->kernel == 3 && !(d->flags & RK_PLAN_NO_SIDE_PAIRS))
      for (size_t k = pairs.size(); k > 0 && pairs[k - 1].first <= rk::kSideMaxTiles; --k)
        ++p->side_pairs;
    info.side_pairs = p->side_pairs;
    // the same pairs grouped by the row range of their last computed row
    // (a pair spans at most a few hundred rows, so with ranges of >= 1024
    // rows it touches only its own range and the one before)
    constexpr int NC = rk_seg_attn_plan_s::kHostChunks;
    p->chunk_rows = std::max<int64_t>(1024, (((rows_total + NC - 1) / NC) + 255) / 256 * 256);
    auto last_row = [&](const TcPair& pr) {
      int64_t last = -1;
      for (int k = 0; k < 2; ++k) {
        const TcTile& t = pr.t[k];
        if (t.pad & 1) continue;
        const DevReq& rq = p->reqs[t.req];
        const int64_t pl = t.kind == 0 ? int64_t(t.p0) + t.p1 - 1 : std::max<int64_t>(t.p0, t.p1);
        last = std::max(last, rq.row_base + (pl - rq.q_row_begin));
      }
      return last;
    };
    std::vector<std::vector<TcPair>> byc(NC);
    for (const TcPair& pr : p->tc_pairs)
      byc[std::min<int64_t>(NC - 1, last_row(pr) / p->chunk_rows)].push_back(pr);
    p->chunk_pair_begin[0] = 0;
    for (int c = 0; c < NC; ++c) {
      for (const TcPair& pr : byc[c]) p->tc_pairs_chunked.push_back(pr);
      p->chunk_pair_begin[c + 1] = static_cast<int32_t>(p->tc_pairs_chunked.size());
    }
    if (p->tc_pairs.size() > (INT32_MAX / 8)) return RK_ERR_CAPACITY;
  } else {
    std::stable_sort(tc_list.begin(), tc_list.end(),
                     [](const auto& a, const auto& b) { return a.first > b.first; });
    for (auto& t : tc_list) {
      info.performed_pairs += t.first * TN * TM;
      p->tc_tiles.push_back(t.second);
    }
    if (p->tc_tiles.size() > (INT32_MAX / 4)) return RK_ERR_CAPACITY;
  }
  info.split_chunks = static_cast<int64_t>(p->chunks.size());
  p->num_parts = parts;
  p->num_mgroups = mgroups;
  size_t wbytes = 0;
  if (parts) {
    const size_t dv = p->d_v;
    size_t bytes = 0;
    bytes += static_cast<size_t>(parts) * kSplitHeads * dv * sizeof(float);
    bytes += static_cast<size_t>(parts) * kSplitHeads * sizeof(float);
    bytes = (bytes + 255) & ~size_t(255);
    bytes += static_cast<size_t>(mgroups) * sizeof(int32_t);
    wbytes = (bytes + 255) & ~size_t(255);
  }
  // the 4-CTA kernel's work queues: one per launch that may run at once
  // (the host-buffer forward launches one per row range)
  p->queue_off = wbytes;
  if (p->kernel == 3 && !p->tc_pairs.empty())
    wbytes += static_cast<size_t>(rk_seg_attn_plan_s::kHostChunks) * rk::kQueueBytes;
  p->workspace_bytes = wbytes;
  return RK_OK;
}

extern "C" rk_status_t rk_seg_attn_plan(const rk_seg_attn_desc_t* desc, void* stream,
                                        rk_seg_attn_plan_t* out) {
  if (!out) return RK_ERR_NULL;
  *out = nullptr;
  if (!desc) return RK_ERR_NULL;
  rk_seg_attn_plan_s* p = new (std::nothrow) rk_seg_attn_plan_s();
  if (!p) return RK_ERR_CAPACITY;
  rk_status_t st = build_plan(desc, p);
  if (st != RK_OK) {
    delete p;
    return st;
  }
  if (!p->host_only) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaGetDevice(&p->device) != cudaSuccess) st = RK_ERR_CUDA;
    if (st == RK_OK) st = upload(p->segs, &p->d_segs, s);
    if (st == RK_OK) st = upload(p->reqs, &p->d_reqs, s);
    if (st == RK_OK) st = upload(p->rope_cs, &p->d_rope_cs, s);
    if (st == RK_OK) st = upload(p->pos_cs_hi, &p->d_pos_cs_hi, s);
    if (st == RK_OK) st = upload(p->pos_cs_lo, &p->d_pos_cs_lo, s);
    if (st == RK_OK) st = upload(p->tiles, &p->d_tiles, s);
    if (st == RK_OK) st = upload(p->local_rows, &p->d_local_rows, s);
    if (st == RK_OK) st = upload(p->global_heads, &p->d_global_heads, s);
    if (st == RK_OK) st = upload(p->local_heads, &p->d_local_heads, s);
    if (st == RK_OK) st = upload(p->chunks, &p->d_chunks, s);
    if (st == RK_OK) st = upload(p->tc_tiles, &p->d_tc_tiles, s);
    if (st == RK_OK) st = upload(p->tc_pairs, &p->d_tc_pairs, s);
    if (st == RK_OK) st = upload(p->tc_pairs_chunked, &p->d_tc_pairs_chunked, s);
    if (st == RK_OK) st = upload(p->head_role, &p->d_head_role, s);
    if (st == RK_OK && p->kernel == 4) {
      // small heads: map 0 of each segment is the latent as [n, d_k]
      // row-major, box 64 dims x 128 rows (dims past d_k read as zero)
      p->segmaps.resize(rk::kSegMaps * p->segs.size());
      const uint64_t dk = static_cast<uint64_t>(p->d_nope + p->d_rope);
      for (size_t i = 0; i < p->segs.size() && st == RK_OK; ++i) {
        const uint64_t dims[2] = {dk, static_cast<uint64_t>(p->segs[i].n)};
        const uint64_t strides[1] = {dk * 2};
        const uint32_t box[2] = {64, 128};
        if (!rk::make_tmap_bf16(&p->segmaps[rk::kSegMaps * i], p->segs[i].latent, 2, dims,
                                strides, box))
          st = RK_ERR_CUDA;
      }
      if (st == RK_OK) st = upload(p->segmaps, &p->d_segmaps, s);
    }
    if (st == RK_OK && p->kernel >= 1 && p->kernel <= 3) {
      // TMA maps of each segment latent, viewing a row as d_k / 64 chunks
      // of 64 bf16: (64, n, d_k / 64) so that a box lands chunk-major in
      // shared memory; map 4 takes whole rows
      p->segmaps.resize(rk::kSegMaps * p->segs.size());
      const uint32_t nch = static_cast<uint32_t>((p->d_nope + p->d_rope) / 64);
      for (size_t i = 0; i < p->segs.size() && st == RK_OK; ++i) {
        const uint64_t dims[3] = {64, static_cast<uint64_t>(p->segs[i].n), nch};
        const uint64_t strides[2] = {static_cast<uint64_t>(nch) * 128, 128};
        const uint32_t boxes[rk::kSegMaps][3] = {
            {64, 128, 2}, {64, 128, 1}, {64, 64, 4}, {64, 64, 1}, {64, 64, nch}, {64, 128, 4}};
        for (int b = 0; b < rk::kSegMaps && st == RK_OK; ++b)
          if (!rk::make_tmap_bf16(&p->segmaps[rk::kSegMaps * i + b], p->segs[i].latent, 3, dims,
                                  strides, boxes[b]))
            st = RK_ERR_CUDA;
      }
      if (st == RK_OK) st = upload(p->segmaps, &p->d_segmaps, s);
    }
    if (st == RK_OK && !p->chunks.empty() && p->d_rope == 64 &&
        (p->d_nope == 512 || (p->v_rope && p->d_nope == 448)) &&
        !(desc->flags & RK_PLAN_LEGACY_MMA)) {
      // split-over-segments chunks stream 32-row boxes of whole latent rows
      const uint32_t nch = static_cast<uint32_t>((p->d_nope + p->d_rope) / 64);
      p->decmaps.resize(p->segs.size());
      for (size_t i = 0; i < p->segs.size() && st == RK_OK; ++i) {
        const uint64_t dims[3] = {64, static_cast<uint64_t>(p->segs[i].n), nch};
        const uint64_t strides[2] = {static_cast<uint64_t>(nch) * 128, 128};
        const uint32_t box[3] = {64, 32, nch};
        if (!rk::make_tmap_bf16(&p->decmaps[i], p->segs[i].latent, 3, dims, strides, box))
          st = RK_ERR_CUDA;
      }
      if (st == RK_OK) st = upload(p->decmaps, &p->d_decmaps, s);
    }
    if (st == RK_OK) {
      if (cudaMalloc(reinterpret_cast<void**>(&p->d_status), sizeof(int32_t)) != cudaSuccess)
        st = RK_ERR_CUDA;
      else if (cudaMemsetAsync(p->d_status, 0, sizeof(int32_t), s) != cudaSuccess)
        st = RK_ERR_CUDA;
    }
    if (st == RK_OK && ((!p->chunks.empty() &&
                         (!p->tiles.empty() || !p->tc_tiles.empty() || !p->tc_pairs.empty())) ||
                        p->side_pairs > 0)) {
      if (cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming) != cudaSuccess)
        st = RK_ERR_CUDA;
    }
    if (st == RK_OK) {
      bool okc = cudaStreamCreateWithFlags(&p->copy_in, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaStreamCreateWithFlags(&p->copy_out, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaStreamCreateWithFlags(&p->compute2, cudaStreamNonBlocking) == cudaSuccess;
      for (cudaEvent_t* e : {&p->ev_start, &p->ev_split, &p->ev_done, &p->ev_c2})
        okc = okc && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
      for (int c = 0; c < rk_seg_attn_plan_s::kHostChunks && okc; ++c)
        okc = cudaEventCreateWithFlags(&p->ev_in[c], cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->ev_k[c], cudaEventDisableTiming) == cudaSuccess;
      if (!okc) st = RK_ERR_CUDA;
    }
    // the side kernel is loaded here: a lazy load at the first forward could
    // wait for the 4-CTA kernel launched just before it to finish
    if (st == RK_OK && p->side_pairs > 0 && rk::prepare_dense_side() != cudaSuccess)
      st = RK_ERR_CUDA;
    // host vectors are pageable: make the uploads complete before returning
    if (st == RK_OK && cudaStreamSynchronize(s) != cudaSuccess) st = RK_ERR_CUDA;
    if (st != RK_OK) {
      free_device(p);
      delete p;
      return st;
    }
  }
  *out = p;
  return RK_OK;
}

extern "C" void rk_seg_attn_plan_destroy(rk_seg_attn_plan_t p) {
  if (!p) return;
  if (!p->host_only) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device) cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    free_device(p);
    if (cur != p->device && cur >= 0) cudaSetDevice(cur);
  }
  delete p;
}

extern "C" rk_status_t rk_seg_attn_plan_info(rk_seg_attn_plan_t p, rk_plan_info_t* info) {
  if (!p || !info) return RK_ERR_NULL;
  *info = p->info;
  return RK_OK;
}

extern "C" int64_t rk_seg_attn_plan_pairs(rk_seg_attn_plan_t p, int32_t* out, int64_t capacity) {
  if (!p) return -1;
  static_assert(sizeof(TcPair) == RK_PAIR_WORDS * sizeof(int32_t), "pair record");
  const int64_t n = static_cast<int64_t>(p->tc_pairs.size());
  const int64_t m = std::min(n, std::max<int64_t>(capacity, 0));
  if (m > 0 && out) std::memcpy(out, p->tc_pairs.data(), static_cast<size_t>(m) * sizeof(TcPair));
  return n;
}

extern "C" size_t rk_seg_attn_workspace_bytes(rk_seg_attn_plan_t p) {
  return p ? p->workspace_bytes : 0;
}

namespace rk {

rk_status_t bind_workspace(const rk_seg_attn_plan_s& p, KernelArgs& a, void* workspace,
                           cudaStream_t s) {
  char* w = static_cast<char*>(workspace);
  if (p.num_parts) {
    a.ws_o = reinterpret_cast<float*>(w);
    size_t off = static_cast<size_t>(p.num_parts) * kSplitHeads * p.d_v * sizeof(float);
    a.ws_lse = reinterpret_cast<float*>(w + off);
    off += static_cast<size_t>(p.num_parts) * kSplitHeads * sizeof(float);
    off = (off + 255) & ~size_t(255);
    a.ws_ticket = reinterpret_cast<int32_t*>(w + off);
    if (cudaMemsetAsync(a.ws_ticket, 0, p.num_mgroups * sizeof(int32_t), s) != cudaSuccess)
      return RK_ERR_CUDA;
  }
  if (p.kernel == 3 && !p.tc_pairs.empty()) {
    a.wq = reinterpret_cast<unsigned long long*>(w + p.queue_off);
    const size_t qb = static_cast<size_t>(rk_seg_attn_plan_s::kHostChunks) * kQueueBytes;
    if (cudaMemsetAsync(a.wq, 0, qb, s) != cudaSuccess) return RK_ERR_CUDA;
  }
  return RK_OK;
}

}  // namespace rk

namespace {

rk_status_t check_forward_args(const rk_seg_attn_plan_s* p, const void* q, const void* out,
                               const float* lse, const void* workspace, size_t ws_bytes) {
  if (!p || !q || !out || !lse) return RK_ERR_NULL;
  if (p->host_only) return RK_ERR_PLAN_MISMATCH;
  auto mis = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) != 0; };
  if (mis(q) || mis(out) || (reinterpret_cast<uintptr_t>(lse) & 3)) return RK_ERR_ALIGNMENT;
  if (p->workspace_bytes) {
    if (!workspace || ws_bytes < p->workspace_bytes) return RK_ERR_WORKSPACE;
    if (mis(workspace)) return RK_ERR_ALIGNMENT;
  }
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return RK_ERR_CUDA;
  if (cur != p->device) return RK_ERR_PLAN_MISMATCH;
  return RK_OK;
}

}  // namespace

extern "C" rk_status_t rk_seg_attn_forward(rk_seg_attn_plan_t p, const void* q, void* out,
                                           float* lse, void* workspace, size_t ws_bytes,
                                           void* stream) {
  rk_status_t st = check_forward_args(p, q, out, lse, workspace, ws_bytes);
  if (st != RK_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rk::KernelArgs a{};
  rk::fill_args(*p, a, q, out, lse);
  st = rk::bind_workspace(*p, a, workspace, s);
  if (st != RK_OK) return st;
  return rk::launch_forward(*p, a, q, s) == cudaSuccess ? RK_OK : RK_ERR_CUDA;
}

extern "C" rk_status_t rk_seg_attn_forward_host(rk_seg_attn_plan_t p, const void* q_host,
                                                void* out_host, float* lse_host, void* q,
                                                void* out, float* lse, void* workspace,
                                                size_t ws_bytes, void* stream) {
  if (!q_host || !out_host || !lse_host) return RK_ERR_NULL;
  rk_status_t st = check_forward_args(p, q, out, lse, workspace, ws_bytes);
  if (st != RK_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  constexpr int NC = rk_seg_attn_plan_s::kHostChunks;
  const int64_t rows = p->info.rows, H = p->H;
  const size_t qrow = static_cast<size_t>(H) * (p->d_nope + p->d_rope) * 2;
  const size_t orow = static_cast<size_t>(H) * p->d_v * 2, lrow = static_cast<size_t>(H) * 4;
  const int64_t CR = p->chunk_rows > 0 ? p->chunk_rows : rows;
  auto range = [&](int c, int64_t& r0, int64_t& r1) {
    r0 = std::min<int64_t>(rows, c * CR);
    r1 = c == NC - 1 ? rows : std::min<int64_t>(rows, (c + 1) * CR);
  };
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  const char* qh = static_cast<const char*>(q_host);
  char* oh = static_cast<char*>(out_host);
  char* lh = reinterpret_cast<char*>(lse_host);
  char* qd = static_cast<char*>(q);
  char* od = static_cast<char*>(out);
  char* ld = reinterpret_cast<char*>(lse);
  // the copies start after the caller's earlier work on s
  bool good = ok(cudaEventRecord(p->ev_start, s)) &&
              ok(cudaStreamWaitEvent(p->copy_in, p->ev_start, 0)) &&
              ok(cudaStreamWaitEvent(p->copy_out, p->ev_start, 0));
  for (int c = 0; c < NC && good; ++c) {
    int64_t r0, r1;
    range(c, r0, r1);
    if (r1 > r0) {
      // q and lse go in; out does not (no kernel reads it)
      const int64_t n = r1 - r0;
      good = ok(cudaMemcpyAsync(qd + r0 * qrow, qh + r0 * qrow, n * qrow, cudaMemcpyHostToDevice,
                                p->copy_in)) &&
             ok(cudaMemcpyAsync(ld + r0 * lrow, lh + r0 * lrow, n * lrow, cudaMemcpyHostToDevice,
                                p->copy_in));
    }
    good = good && ok(cudaEventRecord(p->ev_in[c], p->copy_in));
  }
  rk::KernelArgs a{};
  rk::fill_args(*p, a, q, out, lse);
  if (good) good = rk::bind_workspace(*p, a, workspace, s) == RK_OK;
  const bool pipelined = !p->tc_pairs_chunked.empty() && a.num_tiles == 0 && a.num_tc_tiles == 0;
  if (pipelined) {
    // the tile pairs of row range c run once rows 0 .. c are on the device;
    // the ranges alternate between the caller's stream and a second
    // plan-owned stream, so one range's tiles start on the SMs that the
    // previous range's longest tiles leave idle (the ranges' pairs write
    // disjoint tiles)
    good = good && ok(cudaStreamWaitEvent(p->compute2, p->ev_start, 0));
    for (int c = 0; c < NC && good; ++c) {
      cudaStream_t cs = (c & 1) ? p->compute2 : s;
      good = ok(cudaStreamWaitEvent(cs, p->ev_in[c], 0));
      const int32_t b = p->chunk_pair_begin[c], e = p->chunk_pair_begin[c + 1];
      if (good && e > b) {
        rk::KernelArgs ac = a;
        ac.tc_pairs = p->d_tc_pairs_chunked + b;
        ac.num_tc_pairs = e - b;
        ac.num_chunks = 0;
        ac.num_side_pairs = 0;  // the ranges' pairs run on the 4-CTA clusters alone
        if (a.wq) ac.wq = a.wq + static_cast<size_t>(c) * (rk::kQueueBytes / 8);  // a queue per range
        good = ok(p->kernel == 3 ? rk::launch_dense_tc4(*p, ac, q, cs)
                                 : rk::launch_dense_tc2(*p, ac, q, cs));
      }
      good = good && ok(cudaEventRecord(p->ev_k[c], cs));
    }
    good = good && ok(cudaEventRecord(p->ev_c2, p->compute2)) &&
           ok(cudaStreamWaitEvent(s, p->ev_c2, 0));
    if (good && a.num_chunks) {
      rk::KernelArgs ac = a;
      ac.num_tc_pairs = 0;
      good = ok(rk::launch_split_decode(*p, ac, s));
    }
  } else {
    good = good && ok(cudaStreamWaitEvent(s, p->ev_in[NC - 1], 0)) &&
           ok(rk::launch_forward(*p, a, q, s));
    for (int c = 0; c < NC && good; ++c) good = ok(cudaEventRecord(p->ev_k[c], s));
  }
  good = good && ok(cudaEventRecord(p->ev_split, s));
  // Only the elements the kernels write come back: whole rows where every
  // head is written (protected rows; every row when all heads are Global)
  // and the Global heads' columns of the other rows; the host keeps the rest
  // of out_host as it was.  lse comes back whole (it went in whole).
  const int HG = static_cast<int>(p->global_heads.size());
  const bool all_global = p->local_heads.empty();
  const size_t hbytes = static_cast<size_t>(p->d_v) * 2;
  // Global heads c0 + s g (g < H / s) are one strided copy per range;
  // otherwise one copy per run of consecutive Global heads
  int gstride = 0;
  if (HG > 0 && !all_global && p->H % HG == 0) {
    const int sdiv = p->H / HG;
    bool ev = p->global_heads[0] < sdiv;
    for (int g = 0; g < HG && ev; ++g) ev = p->global_heads[g] == p->global_heads[0] + sdiv * g;
    if (ev) gstride = sdiv;
  }
  size_t run = 0;  // first run of full rows not yet copied
  // range c is final once the kernels of ranges c and c + 1 (and any split
  // chunks) are done
  for (int c = 0; c < NC && good; ++c) {
    int64_t r0, r1;
    range(c, r0, r1);
    good = ok(cudaStreamWaitEvent(p->copy_out, p->ev_k[c], 0)) &&
           ok(cudaStreamWaitEvent(p->copy_out, p->ev_k[std::min(c + 1, NC - 1)], 0));
    if (good && a.num_chunks) good = ok(cudaStreamWaitEvent(p->copy_out, p->ev_split, 0));
    if (!good || r1 <= r0) continue;
    const int64_t n = r1 - r0;
    good = ok(cudaMemcpyAsync(lh + r0 * lrow, ld + r0 * lrow, n * lrow, cudaMemcpyDeviceToHost,
                              p->copy_out));
    if (all_global) {
      good = good && ok(cudaMemcpyAsync(oh + r0 * orow, od + r0 * orow, n * orow,
                                        cudaMemcpyDeviceToHost, p->copy_out));
      continue;
    }
    if (good && gstride > 0) {
      const size_t off = r0 * orow + p->global_heads[0] * hbytes;
      good = ok(cudaMemcpy2DAsync(oh + off, gstride * hbytes, od + off, gstride * hbytes, hbytes,
                                  static_cast<size_t>(n) * HG, cudaMemcpyDeviceToHost,
                                  p->copy_out));
    } else {
      for (int g = 0; g < HG && good;) {
        int e = g + 1;
        while (e < HG && p->global_heads[e] == p->global_heads[e - 1] + 1) ++e;
        const size_t off = r0 * orow + p->global_heads[g] * hbytes;
        good = ok(cudaMemcpy2DAsync(oh + off, orow, od + off, orow, (e - g) * hbytes,
                                    static_cast<size_t>(n), cudaMemcpyDeviceToHost, p->copy_out));
        g = e;
      }
    }
    while (good && run < p->full_rows.size() && p->full_rows[run].first < r1) {
      const int64_t f0 = std::max(r0, p->full_rows[run].first);
      const int64_t f1 = std::min(r1, p->full_rows[run].second);
      if (f1 > f0)
        good = ok(cudaMemcpyAsync(oh + f0 * orow, od + f0 * orow, (f1 - f0) * orow,
                                  cudaMemcpyDeviceToHost, p->copy_out));
      if (p->full_rows[run].second > r1) break;  // continues in the next range
      ++run;
    }
  }
  // the caller's stream resumes when everything is back on the host
  good = good && ok(cudaEventRecord(p->ev_done, p->copy_out)) &&
         ok(cudaStreamWaitEvent(s, p->ev_done, 0));
  return good ? RK_OK : RK_ERR_CUDA;
}

namespace rk {

void fill_args(const rk_seg_attn_plan_s& p, KernelArgs& a, const void* q, void* out, float* lse) {
  a.q = static_cast<const uint16_t*>(q);
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.segs = p.d_segs;
  a.reqs = p.d_reqs;
  a.rope_cs = p.d_rope_cs;
  a.tiles = p.d_tiles;
  a.num_tiles = static_cast<int32_t>(p.tiles.size());
  a.local_rows = p.d_local_rows;
  a.global_heads = p.d_global_heads;
  a.local_heads = p.d_local_heads;
  a.num_global = static_cast<int32_t>(p.global_heads.size());
  a.num_local = static_cast<int32_t>(p.local_heads.size());
  a.H = p.H;
  a.sink = p.sink;
  a.window = p.window;
  a.scale_log2 = p.softmax_scale * 1.4426950408889634f;
  a.chunks = p.d_chunks;
  a.num_chunks = static_cast<int32_t>(p.chunks.size());
  a.status = p.d_status;
  a.tc_tiles = p.d_tc_tiles;
  a.num_tc_tiles = static_cast<int32_t>(p.tc_tiles.size());
  a.rows_per_gtile = p.global_heads.empty() ? 0 : kTcM / static_cast<int>(p.global_heads.size());
  a.segmaps = p.d_segmaps;
  a.head_role = p.d_head_role;
  a.g_ingroup = p.g_ingroup;
  a.decmaps = p.d_decmaps;
  a.tc_pairs = p.d_tc_pairs;
  a.num_tc_pairs = static_cast<int32_t>(p.tc_pairs.size());
  a.v_rope = p.v_rope ? 1 : 0;
  a.d_v = p.d_v;
  a.pos_cs_hi = p.d_pos_cs_hi;
  a.pos_cs_lo = p.d_pos_cs_lo;
  a.num_side_pairs = p.side_pairs;
}

cudaError_t launch_forward(const rk_seg_attn_plan_s& p, const KernelArgs& a, const void* q,
                           cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  // prefill tiles overlap the split chunks on the plan's side stream
  cudaStream_t ts = s;
  if (p.side && a.num_chunks && (a.num_tiles || a.num_tc_tiles || a.num_tc_pairs)) {
    e = cudaEventRecord(p.ev_fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.side, p.ev_fork, 0);
    if (e != cudaSuccess) return e;
    ts = p.side;
  }
  if (a.num_tiles) e = p.kernel == 4 ? launch_dense_tcs(p, a, ts) : launch_dense_mma(p, a, ts);
  if (e == cudaSuccess && a.num_tc_tiles) e = launch_dense_tc(p, a, q, ts);
  // beside split chunks (decode) the few short Local tiles run on CTA pairs,
  // which leave more SMs to the split kernel than 4-CTA clusters (the pair
  // kernel has no rotary-value form)
  if (e == cudaSuccess && a.num_tc_pairs) {
    if (p.kernel == 3 && !a.num_chunks && a.num_side_pairs > 0 && p.side) {
      // the 4-CTA clusters first, then the side kernel on the plan's stream
      // (forked before the clusters' launch, so that it runs beside them on
      // the SMs they leave free)
      int64_t clusters = 0;
      e = dense_tc4_clusters(p, a, clusters);
      if (e == cudaSuccess) e = prepare_dense_side();
      if (e == cudaSuccess) e = cudaEventRecord(p.ev_fork, s);
      if (e == cudaSuccess) e = launch_dense_tc4(p, a, q, s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(p.side, p.ev_fork, 0);
      if (e == cudaSuccess) e = launch_dense_side(p, a, q, clusters, p.side);
      if (e == cudaSuccess) e = cudaEventRecord(p.ev_join, p.side);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, p.ev_join, 0);
    } else {
      e = (p.kernel == 3 && (!a.num_chunks || p.v_rope)) ? launch_dense_tc4(p, a, q, ts)
                                                          : launch_dense_tc2(p, a, q, ts);
    }
  }
  if (e == cudaSuccess && a.num_chunks) e = launch_split_decode(p, a, s);
  if (ts != s) {
    const cudaError_t e1 = cudaEventRecord(p.ev_join, ts);
    const cudaError_t e2 = e1 == cudaSuccess ? cudaStreamWaitEvent(s, p.ev_join, 0) : e1;
    if (e == cudaSuccess) e = e2;
  }
  return e;
}

}  // namespace rk

extern "C" rk_status_t rk_lse_merge(const float* o_parts, const float* lse_parts, int32_t P,
                                    int64_t rows, int32_t H, int32_t d_v, void* out,
                                    float* lse_out, void* stream) {
  if (!o_parts || !lse_parts || !out || !lse_out) return RK_ERR_NULL;
  if (P < 1 || rows < 0 || H < 1 || d_v < 1 || d_v > 1024) return RK_ERR_INVALID_ARG;
  if (rows * H > (int64_t(1) << 40)) return RK_ERR_CAPACITY;
  if ((reinterpret_cast<uintptr_t>(o_parts) | reinterpret_cast<uintptr_t>(lse_parts) |
       reinterpret_cast<uintptr_t>(lse_out)) & 3)
    return RK_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(out) & 1) return RK_ERR_ALIGNMENT;
  if (rows == 0) return RK_OK;
  cudaError_t e = rk::launch_lse_merge(o_parts, lse_parts, P, rows, H, d_v,
                                       static_cast<uint16_t*>(out), lse_out,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RK_OK : RK_ERR_CUDA;
}

extern "C" rk_status_t rk_seg_attn_last_device_status(rk_seg_attn_plan_t p, void* stream) {
  if (!p) return RK_ERR_NULL;
  if (p->host_only) return RK_ERR_PLAN_MISMATCH;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, p->d_status, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return RK_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RK_ERR_CUDA;
  if (cudaMemsetAsync(p->d_status, 0, sizeof(int32_t), s) != cudaSuccess) return RK_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RK_ERR_CUDA;
  return h ? static_cast<rk_status_t>(h) : RK_OK;
}
