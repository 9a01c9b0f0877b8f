// Internal types shared by the host plan and the CUDA kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>
#include <vector>

#include "rk_seg_attn.h"

namespace rk {

// TMA maps per segment latent (viewed as (64, n, 9 chunks)), by box:
// 0: 128 rows x 2 chunks, 1: 128 rows x 1 chunk, 2: 64 rows x 4 chunks,
// 3: 64 rows x 1 chunk, 4: 64 rows x 9 chunks, 5: 128 rows x 4 chunks.
constexpr int kSegMaps = 6;

// One segment as the kernels see it; segments of a request are stored
// contiguously, sorted by offset.
struct DevSeg {
  const uint16_t* latent;  // bf16 [n, d_k]
  int32_t n;
  int32_t delta;
  int32_t is_new;
  int32_t pad;
};

struct DevReq {
  int32_t seg_first;   // index of the request's first DevSeg
  int32_t seg_count;
  int32_t T;           // rows of the request
  int32_t q_row_begin; // first computed absolute row
  int64_t row_base;    // flattened computed-row index of q_row_begin
};

// A prefill-style work tile: a set of (row, head) query pairs that share
// one key range.  kind 0: rows [first, first + count) x every Global head.
// kind 1: pairs [first, first + count) of the flattened (protected row,
// Local head) list, pair i -> (local_rows[i / HL], local_heads[i % HL]).
// Keys visited: [0, sink_hi) u [win_lo, key_hi), clipped to each segment.
struct DenseTile {
  int32_t req;
  int32_t kind;
  int32_t first;
  int32_t count;
  int32_t key_hi;
  int32_t win_lo;
  int32_t sink_hi;
  int32_t pad;
};

// A split-over-segments chunk (single computed row, Global heads): keys
// [k0, k1) (absolute) inside segment `seg`, head group `group` (8 Global
// heads), partial slot `part` of the merge group `mgroup` whose parts are
// [part_first, part_first + nparts).
struct SplitChunk {
  int32_t req;
  int32_t seg;       // global DevSeg index
  int32_t k0, k1;
  int32_t group;
  int32_t part;
  int32_t mgroup;
  int32_t part_first;
  int32_t nparts;
  int32_t pad[3];
};

// A tile of the tcgen05 kernel: 128 query pairs.  kind 0: rows
// [p0, p0 + p1) x every Global head (128 / HG rows per tile, head-major).
// kind 1: protected rows p0 and p1 (p1 < 0: none) x every head (128 / H rows
// per tile, row-major); only the Local heads are stored.  Keys visited:
// [0, sink_hi) u [win_lo, key_hi).  Each tile runs on two CTAs, one per half
// of d_v.
struct TcTile {
  int32_t req;
  int32_t kind;
  int32_t p0;
  int32_t p1;
  int32_t key_hi;
  int32_t win_lo;
  int32_t sink_hi;
  int32_t pad;
};

// Two tcgen05 tiles of one request run as a CTA pair (cta_group::2) over
// the union of their key ranges, [0, sink_hi) u [win_lo, key_hi) with
// sink_hi <= win_lo.  t[1].pad bit 0 marks a partner without work (its CTA
// computes on a copy of t[0] and stores nothing).  Each pair runs on four
// CTAs: two per half of d_v.  `skip` packs the request's segments
// [skip & 0xffff, skip >> 16) that lie wholly between the two key ranges
// (0 = none), for the key walk to jump over.
struct TcPair {
  TcTile t[2];
  int32_t key_hi;
  int32_t win_lo;
  int32_t sink_hi;
  int32_t skip;
};

// Work queue of one launch of the persistent 4-CTA kernel and of the side
// kernel beside it: a 64-bit claim counter (word 0: the pairs taken from the
// front of the list in its low half, from the back in its high half) and,
// from word 32 on, a ring of kQueueRing claimed items for each of up to
// kQueueClusters 4-CTA clusters and kSideClusters side CTA pairs.
constexpr int kQueueClusters = 40;
constexpr int kSideClusters = 8;
constexpr int kQueueRing = 64;
constexpr size_t kQueueBytes =
    256 + static_cast<size_t>(kQueueClusters + kSideClusters) * kQueueRing * 8;
// the side kernel takes only pairs of at most this many key tiles
constexpr int kSideMaxTiles = 8;

struct KernelArgs {
  const uint16_t* q;
  uint16_t* out;
  float* lse;
  const DevSeg* segs;
  const DevReq* reqs;
  const float* rope_cs;       // [num_segs][d_rope/2][2] cos, sin of delta * theta
  const DenseTile* tiles;
  int32_t num_tiles;
  const int32_t* local_rows;  // compacted protected computed rows (absolute)
  const int32_t* global_heads;
  const int32_t* local_heads;
  int32_t num_global, num_local;
  int32_t H;
  int32_t sink, window;
  float scale_log2;           // softmax_scale * log2(e)
  const SplitChunk* chunks;
  int32_t num_chunks;
  float* ws_o;                // [parts][8][d_v]
  float* ws_lse;              // [parts][8]
  int32_t* ws_ticket;         // [mgroups]
  int32_t* status;            // device status word
  const TcTile* tc_tiles;
  int32_t num_tc_tiles;
  int32_t rows_per_gtile;     // 128 / HG
  const CUtensorMap* segmaps; // kSegMaps per segment
  const uint8_t* head_role;   // [H]
  int32_t g_ingroup;          // Global heads are 8g + g_ingroup for every group g, or -1
  const CUtensorMap* decmaps; // per segment: latent viewed (64, n, d_k / 64 chunks), box 32 rows x all chunks
  const TcPair* tc_pairs;
  int32_t num_tc_pairs;
  int32_t v_rope;             // V is the whole latent row (d_v = d_k), output phase restored
  int32_t d_v;                // output columns
  const float* pos_cs_hi;     // [T / 256 + 1][d_rope/2][2] cos, sin of 256 a theta   (v_rope)
  const float* pos_cs_lo;     // [256][d_rope/2][2] cos, sin of b theta              (v_rope)
  unsigned long long* wq;     // work queue of the 4-CTA kernel (kQueueBytes, zeroed)
  int32_t num_side_pairs;     // the short tail of tc_pairs that the side kernel may take
};

}  // namespace rk

struct rk_seg_attn_plan_s {
  int device = -1;
  bool host_only = false;
  int32_t H = 0, d_nope = 0, d_rope = 0;
  int32_t d_v = 0;
  bool v_rope = false;
  int32_t sink = 0, window = 0;
  float softmax_scale = 0.f;
  int kernel = 0;          // 0 mma.sync, 1 tcgen05 tiles, 2 CTA-pair tiles, 3 4-CTA tiles
  int tile_m = 64;         // query pairs per dense tile
  int g_ingroup = -1;      // Global heads are exactly 8g + g_ingroup, else -1
  rk_plan_info_t info{};
  // host copies
  std::vector<rk::DevSeg> segs;
  std::vector<rk::DevReq> reqs;
  std::vector<float> rope_cs;
  std::vector<float> pos_cs_hi, pos_cs_lo;
  std::vector<rk::DenseTile> tiles;
  std::vector<int32_t> local_rows;
  // runs [first, end) of flattened computed rows whose every head is written
  // (protected rows); the host forward copies back these rows whole and only
  // the Global heads of the others
  std::vector<std::pair<int64_t, int64_t>> full_rows;
  std::vector<int32_t> global_heads, local_heads;
  std::vector<rk::SplitChunk> chunks;
  std::vector<rk::TcTile> tc_tiles;
  std::vector<rk::TcPair> tc_pairs;
  std::vector<CUtensorMap> segmaps;
  std::vector<CUtensorMap> decmaps;
  std::vector<uint8_t> head_role;
  int64_t num_parts = 0;
  int64_t num_mgroups = 0;
  // device copies
  rk::DevSeg* d_segs = nullptr;
  rk::DevReq* d_reqs = nullptr;
  float* d_rope_cs = nullptr;
  float* d_pos_cs_hi = nullptr;
  float* d_pos_cs_lo = nullptr;
  rk::DenseTile* d_tiles = nullptr;
  int32_t* d_local_rows = nullptr;
  int32_t* d_global_heads = nullptr;
  int32_t* d_local_heads = nullptr;
  rk::SplitChunk* d_chunks = nullptr;
  rk::TcTile* d_tc_tiles = nullptr;
  rk::TcPair* d_tc_pairs = nullptr;
  CUtensorMap* d_segmaps = nullptr;
  CUtensorMap* d_decmaps = nullptr;
  uint8_t* d_head_role = nullptr;
  int32_t* d_status = nullptr;
  size_t workspace_bytes = 0;
  size_t queue_off = 0;       // the 4-CTA kernel's work queues (kHostChunks of kQueueBytes)
  int32_t side_pairs = 0;     // pairs at the end of tc_pairs with <= kSideMaxTiles key tiles
  // when a forward has both split chunks and prefill tiles, the tiles run on
  // this plan-owned stream, forked from and joined back to the caller's; a
  // forward on 4-CTA clusters runs the side kernel there
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // forward from host buffers: the computed rows in kHostChunks ranges of
  // chunk_rows rows, the tile pairs grouped by the range of their last row
  // (each group longest first), and the streams and events that overlap the
  // copies of one range with the kernels of another
  static constexpr int kHostChunks = 8;
  int64_t chunk_rows = 0;
  std::vector<rk::TcPair> tc_pairs_chunked;
  int32_t chunk_pair_begin[kHostChunks + 1] = {};
  rk::TcPair* d_tc_pairs_chunked = nullptr;
  cudaStream_t copy_in = nullptr, copy_out = nullptr, compute2 = nullptr;
  cudaEvent_t ev_start = nullptr, ev_split = nullptr, ev_done = nullptr, ev_c2 = nullptr;
  cudaEvent_t ev_in[kHostChunks] = {}, ev_k[kHostChunks] = {};
};

namespace rk {
// Kernel launchers (defined in the .cu files).
cudaError_t launch_dense_mma(const rk_seg_attn_plan_s& plan, const KernelArgs& a,
                             cudaStream_t stream);
cudaError_t launch_split_decode(const rk_seg_attn_plan_s& plan, const KernelArgs& a,
                                cudaStream_t stream);
cudaError_t launch_dense_tc(const rk_seg_attn_plan_s& plan, const KernelArgs& a,
                            const void* q, cudaStream_t stream);
cudaError_t launch_dense_tc2(const rk_seg_attn_plan_s& plan, const KernelArgs& a,
                             const void* q, cudaStream_t stream);
cudaError_t launch_dense_tc4(const rk_seg_attn_plan_s& plan, const KernelArgs& a,
                             const void* q, cudaStream_t stream);
// 4-CTA clusters that launch_dense_tc4 starts for these arguments.
cudaError_t dense_tc4_clusters(const rk_seg_attn_plan_s& plan, const KernelArgs& a,
                               int64_t& clusters);
// The side kernel: persistent CTA pairs on the SMs that `tc4_clusters`
// 4-CTA clusters leave free, taking the short pairs from the back of the
// same work queue (none launched when no SM pair is free).
cudaError_t launch_dense_side(const rk_seg_attn_plan_s& plan, const KernelArgs& a,
                              const void* q, int64_t tc4_clusters, cudaStream_t stream);
// Sets the side kernel's attributes.  With lazy module loading the first
// such call loads the kernel, which may wait for the device to go idle, so
// it is made before the 4-CTA kernel is launched.
cudaError_t prepare_dense_side();
cudaError_t launch_dense_tcs(const rk_seg_attn_plan_s& plan, const KernelArgs& a,
                             cudaStream_t stream);
// Fill the kernel arguments shared by every launch of a forward.
void fill_args(const rk_seg_attn_plan_s& plan, KernelArgs& a, const void* q, void* out,
               float* lse);
// Point the split-decode arguments at `workspace` (the layout that
// rk_seg_attn_workspace_bytes sizes: partial outputs, partial LSEs, then the
// merge tickets at a 256-byte boundary) and clear the tickets on stream s.
rk_status_t bind_workspace(const rk_seg_attn_plan_s& plan, KernelArgs& a, void* workspace,
                           cudaStream_t s);
// Launch every kernel of a forward (split chunks, then prefill tiles).
cudaError_t launch_forward(const rk_seg_attn_plan_s& plan, const KernelArgs& a, const void* q,
                           cudaStream_t stream);
cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int32_t P,
                             int64_t rows, int32_t H, int32_t d_v, uint16_t* out,
                             float* lse_out, cudaStream_t stream);
}  // namespace rk
