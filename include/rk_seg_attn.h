/*
 * rk_seg_attn.h - C ABI of the segment-relocated MLA attention library.
 *
 * The operation is the online attention step of RedKnot-MLA (arXiv
 * 2609.07008, "RedKnot-MLA: Multi-Head Offline-Online Reuse for DeepSeek-V4
 * Long-Context Serving"):
 *
 *   - every immutable document i is a canonical packed MLA latent C_i built
 *     alone at positions 0..n_i-1 (artifacts paragraph) and placed at request
 *     offset delta_i;
 *   - the runtime rotates the query's RoPE slice by -delta_i, attends the
 *     canonical latent in place (K = [c_nope | k_rope], V = c_nope, the one
 *     packed latent shared by every logical head), and combines the
 *     per-segment statistics with a numerically stable log-sum-exp merge
 *     (RoPE-orthogonality paragraph);
 *   - logical heads have two roles (head-partition paragraph, eq. (1)):
 *     Global heads attend causally to the whole request; Local heads see the
 *     sink and the window [p - w, p] only (RedKnot blog "RedKnot, explained",
 *     "Insight 1", window W(i));
 *   - the Local rows of the protected set are replaced by the recomputed
 *     values, never added (protected-set paragraph).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * bf16     IEEE bfloat16 stored as uint16.
 * d_k      d_nope + d_rope;  d_v = d_nope (V = c_nope), or d_v = d_k with
 *          RK_PLAN_V_ROPE (V = the whole latent row, see there).
 * RoPE     interleaved pairs (2j, 2j+1) of the rope slice, theta_j =
 *          rope_base^(-2j/d_rope); R(phi) turns (x, y) into
 *          (x cos - y sin, x sin + y cos) with angle phi * theta_j.
 * rows     The rows a forward computes are, per request r in order, the
 *          absolute positions q_row_begin[r] .. T_r - 1 (T_r = sum of the
 *          request's segment lengths).  Q, out and lse are indexed by this
 *          flattened "computed row" index.
 * scores   x = softmax_scale * q.k; lse is the natural-log LSE of x.
 * streams  `stream` is a cudaStream_t passed as void*; NULL is the legacy
 *          default stream.  Entry points that take a stream enqueue work and
 *          return without synchronising unless stated otherwise.
 * errors   Every argument or geometry error is returned synchronously before
 *          any launch and leaves all buffers untouched.  A failed CUDA call
 *          returns RK_ERR_CUDA.  There is no fallback path of any kind.
 */
#ifndef RK_SEG_ATTN_H
#define RK_SEG_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RK_OK = 0,
  RK_ERR_NULL = 1,              /* a required pointer is NULL */
  RK_ERR_INVALID_ARG = 2,       /* a count, size or value is out of range */
  RK_ERR_SEGMENT_OVERLAP = 3,   /* two segments of a request share a row */
  RK_ERR_SEGMENT_GAP = 4,       /* segments do not tile [0, T_r) */
  RK_ERR_UNSUPPORTED_DIMS = 5,  /* (d_nope, d_rope) not compiled in */
  RK_ERR_CAPACITY = 6,          /* a size exceeds an int32 index or a fixed limit */
  RK_ERR_CUDA = 7,              /* a CUDA runtime/driver call failed */
  RK_ERR_DEVICE_TIMEOUT = 8,    /* a bounded device-side wait expired */
  RK_ERR_PLAN_MISMATCH = 9,     /* the plan was built host-only or for another device */
  RK_ERR_ALIGNMENT = 10,        /* a device pointer is not 16-byte aligned */
  RK_ERR_WORKSPACE = 11         /* workspace missing or smaller than required */
} rk_status_t;

/* Segment flag: the request's own new rows (always protected, causal among
 * themselves like every other row). */
#define RK_SEG_NEW 1u

/* Plan flags. */
#define RK_PLAN_HOST_ONLY 1u    /* build and validate on the host only: no
                                   device memory, forward refuses the plan */
#define RK_PLAN_LEGACY_MMA 2u   /* run the prefill tiles on the mma.sync
                                   kernel instead of a tcgen05 kernel */
#define RK_PLAN_SINGLE_CTA 4u   /* run each tcgen05 tile on its own two CTAs
                                   (one per half of d_v) */
#define RK_PLAN_DEVICE_BITMAP 16u /* protected_bitmap is a device pointer
                                   (e.g. written by rk_protected_build); the
                                   plan copies it to the host */
#define RK_PLAN_CTA_PAIR 8u     /* run pairs of tcgen05 tiles on CTA pairs,
                                   one pair per half of d_v, instead of
                                   4-CTA clusters (scores on one CTA pair,
                                   outputs on the other) */
#define RK_PLAN_NO_SIDE_PAIRS 64u /* run every tile pair on the 4-CTA
                                   clusters.  By default, on a GPU whose SMs
                                   do not divide into 4-CTA clusters, a
                                   persistent CTA-pair kernel on the SMs the
                                   clusters leave free (a second stream, forked
                                   from and joined back to the caller's) takes
                                   the shortest pairs (at most 8 key tiles)
                                   from the back of the same work list, with
                                   the same arithmetic, so the results are the
                                   same either way.  Set this when other work
                                   is meant to use those SMs meanwhile. */
#define RK_PLAN_V_ROPE 32u      /* the value carries a rotary part: V is the
                                   whole packed latent row [c_nope | k_rope]
                                   (d_v = d_k).  Each segment's contribution
                                   to the output's rope slice is moved to
                                   absolute positions by R(+delta_i) before
                                   the merge, and the merged output's rope
                                   slice is turned by the inverse output RoPE
                                   R(-p) at the query row's absolute position
                                   p, so it equals sum_k P_k R(k - p) v_k
                                   (RedKnot-MLA paper: R^-1 in the
                                   head-partition paragraph; "restores the
                                   output phase", RoPE-orthogonality
                                   paragraph).  Requires (d_nope, d_rope) =
                                   (448, 64): the fp32 output accumulator of a
                                   128-row tile fills the 512 columns of
                                   tensor memory.  Runs on the 4-CTA kernel
                                   (H = 64 or 128, one Global head per group
                                   of 8 or none) and the split decode kernel;
                                   RK_PLAN_LEGACY_MMA, RK_PLAN_SINGLE_CTA and
                                   RK_PLAN_CTA_PAIR are refused with it. */

/* One document segment of a request.
 * latent  device pointer, bf16 [n, d_k] row-major (row stride d_k elements),
 *         16-byte aligned, row j = [c_nope | k_rope] with k_rope rotated at
 *         canonical position j.  Owned by the caller; it must stay valid and
 *         unchanged while any forward using the plan is in flight.
 * n       rows (>= 1).
 * delta   request offset of row 0 (>= 0).
 * flags   0 or RK_SEG_NEW. */
typedef struct {
  const void* latent;
  int64_t n;
  int64_t delta;
  uint32_t flags;
  uint32_t reserved;  /* must be 0 */
} rk_segment_t;

/* Request geometry and head roles.  Every pointer here is a HOST pointer and
 * is only read during rk_seg_attn_plan.
 * num_requests     R >= 1.
 * seg_begin        [R + 1] prefix offsets into segs (seg_begin[0] == 0).
 * segs             segment table, any order within a request; the segments
 *                  of a request must tile [0, T_r) exactly.
 * q_row_begin      [R] first computed row of each request (0 for a prefill
 *                  that recomputes every row; T_r - 1 for a decode step).
 * num_heads        H, a multiple of 8, at most 256.
 * d_nope, d_rope   (512, 64) or (128, 32); (448, 64) with RK_PLAN_V_ROPE.
 * rope_base        theta base (> 1).
 * softmax_scale    s > 0, usually 1/sqrt(d_k).
 * head_role        [H] 0 = Local, 1 = Global.
 * sink, window     Local visibility: keys k <= p with k < sink or k >= p - window.
 * protected_bitmap concatenated per-request bitmaps of ceil(T_r / 32) uint32
 *                  words each, bit p % 32 of word p / 32 (LSB first) set when
 *                  absolute row p is protected; NULL means no protected rows
 *                  besides the RK_SEG_NEW rows, which are always protected.
 * flags            RK_PLAN_* bits. */
typedef struct {
  int32_t num_requests;
  const int32_t* seg_begin;
  const rk_segment_t* segs;
  const int64_t* q_row_begin;
  int32_t num_heads;
  int32_t d_nope;
  int32_t d_rope;
  double rope_base;
  float softmax_scale;
  const uint8_t* head_role;
  int32_t sink;
  int32_t window;
  const uint32_t* protected_bitmap;
  uint32_t flags;
} rk_seg_attn_desc_t;

typedef struct rk_seg_attn_plan_s* rk_seg_attn_plan_t;

/* Host-side counts of a plan (for reports and tests). */
typedef struct {
  int64_t rows;              /* computed rows (leading dimension of q/out/lse) */
  int32_t num_heads, d_nope, d_rope;
  int32_t num_global_heads, num_local_heads;
  int64_t protected_local_rows;   /* computed rows whose Local heads are recomputed */
  int64_t dense_tiles;       /* prefill-style work tiles */
  int64_t split_chunks;      /* split-over-segments chunks (decode) */
  int64_t pairs_global;      /* attended (row, Global head, key) pairs */
  int64_t pairs_local;       /* attended (row, Local head, key) pairs */
  int64_t performed_pairs;   /* M_tile x N_tile summed over issued key tiles */
  int64_t latent_bytes;      /* bytes of every segment latent */
  int32_t kernel;            /* 0 = mma.sync tiles, 1 = tcgen05 tiles,
                                2 = tcgen05 tiles paired on CTA pairs,
                                3 = tcgen05 tile pairs on 4-CTA clusters,
                                4 = tcgen05 tiles for small heads (d_nope 128,
                                    d_rope 32), one CTA per tile */
  int32_t d_v;               /* output columns: d_nope, or d_k with RK_PLAN_V_ROPE */
  int64_t side_pairs;        /* kernel 3: tile pairs at the end of the work list
                                (at most 8 key tiles each) that the side kernel
                                beside the 4-CTA clusters may take (prefill
                                forwards without split decode rows); 0 with
                                RK_PLAN_NO_SIDE_PAIRS */
} rk_plan_info_t;

/* Build an immutable, reusable plan for one request bundle geometry
 * (paper, TP8 fast-path paragraph: repeated document bundles reuse compact
 * segment-pointer geometry).  Validates the descriptor, sorts segments by
 * offset, computes the fp64 cos/sin(delta_i theta_j) table (stored fp32),
 * compacts the protected rows, enumerates the work tiles (fully masked tiles
 * are never listed) longest first, and uploads everything on `stream`.
 * Owns copies of all host inputs; the descriptor may be freed on return.
 * The segment latent pointers are recorded, not copied.
 * Errors: RK_ERR_NULL, RK_ERR_INVALID_ARG, RK_ERR_SEGMENT_OVERLAP,
 * RK_ERR_SEGMENT_GAP, RK_ERR_UNSUPPORTED_DIMS, RK_ERR_CAPACITY,
 * RK_ERR_ALIGNMENT (a latent not 16-byte aligned), RK_ERR_CUDA.  On error
 * *out is set to NULL and nothing is allocated. */
rk_status_t rk_seg_attn_plan(const rk_seg_attn_desc_t* desc, void* stream,
                             rk_seg_attn_plan_t* out);

/* Release a plan (synchronises the device first; NULL is ignored). */
void rk_seg_attn_plan_destroy(rk_seg_attn_plan_t plan);

/* Fill *info with the plan's counts.  Host only; errors: RK_ERR_NULL. */
rk_status_t rk_seg_attn_plan_info(rk_seg_attn_plan_t plan, rk_plan_info_t* info);

/* Diagnostics: the tile pairs of a plan on the 4-CTA prefill kernel (kernel
 * 3), in the plan's order (longest first), RK_PAIR_WORDS int32 per pair:
 *   [0..7]   tile 0: request, kind (0 Global rows x Global heads, 1 one or
 *            two protected rows x every head), p0, p1, key_hi, win_lo,
 *            sink_hi, flags (bit 0: a partner without work)
 *   [8..15]  tile 1, the same
 *   [16..18] the pair's key ranges: key_hi, win_lo, sink_hi (keys
 *            [0, sink_hi) u [win_lo, key_hi), absolute within the request)
 *   [19]     segment skip: the request's segments [skip & 0xffff, skip >> 16)
 *            meet neither range (0: none)
 * Copies min(count, capacity) pairs to `out` (host memory; may be NULL when
 * capacity is 0) and returns the count, or -1 for a NULL plan.  Host only. */
#define RK_PAIR_WORDS 20
int64_t rk_seg_attn_plan_pairs(rk_seg_attn_plan_t plan, int32_t* out, int64_t capacity);

/* Bytes of device workspace rk_seg_attn_forward needs (0 if none): the
 * partial outputs of split decode rows, and for plans on the 4-CTA prefill
 * kernel (kernel 3) the work queues its persistent clusters, and the side
 * kernel beside them, claim tile pairs from (about 199 KB). */
size_t rk_seg_attn_workspace_bytes(rk_seg_attn_plan_t plan);

/* Segment-relocated attention over the plan's segments (paper,
 * RoPE-orthogonality and protected-set paragraphs; blog "Insight 1").
 * q          device bf16 [rows, H, d_k], q_rope rotated at the row's absolute
 *            position, 16-byte aligned.
 * out        device bf16 [rows, H, d_v], in/out.  Global heads: written on
 *            every computed row.  Local heads: written only on protected
 *            rows (bitmap bit set or RK_SEG_NEW row); every other element
 *            keeps its bytes.
 * lse        device fp32 [rows, H], in/out, written exactly where out is.
 * workspace  device scratch of rk_seg_attn_workspace_bytes(plan) bytes,
 *            16-byte aligned (may be NULL when that is 0); its contents on
 *            entry are irrelevant.  Forwards that share a workspace must be
 *            ordered on one stream.
 * Asynchronous on `stream`.  A forward with split decode rows beside
 * prefill tiles, or with the side kernel beside the 4-CTA clusters, forks
 * part of its work onto a plan-owned stream (recorded events order it after
 * the work queued on `stream` before the call, and `stream` continues only
 * after it); forwards on one plan issued from several host threads at once
 * may therefore wait for one another there.  Errors: RK_ERR_NULL,
 * RK_ERR_ALIGNMENT, RK_ERR_WORKSPACE, RK_ERR_PLAN_MISMATCH, RK_ERR_CUDA
 * (launch failure).  Device-side wait expiries are reported by
 * rk_seg_attn_last_device_status. */
rk_status_t rk_seg_attn_forward(rk_seg_attn_plan_t plan, const void* q, void* out,
                                float* lse, void* workspace, size_t workspace_bytes,
                                void* stream);

/* The same forward with q, out and lse starting and ending in host memory:
 * the copies to and from the device run inside the call, overlapped with
 * the kernels.  The computed rows are taken in eight consecutive ranges;
 * a range's q and lse rows are copied in on a plan-owned stream, its tiles
 * run as soon as it (and every earlier range) is on the device, alternately
 * on `stream` and on a second plan-owned stream,
 * and its results are copied back on a third plan-owned stream once the
 * tiles that write it are done.  Only written elements of out travel: the
 * whole row where every head is written (protected rows, or every row when
 * all heads are Global) and the Global heads' columns of the other rows;
 * out is never copied in, since no kernel reads it.
 * (The pages have no counterpart; this is how a host-resident query batch
 * meets the device-resident document latents.)
 * q_host, out_host, lse_host  host arrays of the shapes of q, out, lse
 *            below; out_host and lse_host are in/out exactly like out and
 *            lse.  Page-locked memory lets the copies overlap; pageable
 *            memory is accepted and is copied synchronously.
 * q, out, lse device arrays of the full sizes (as for rk_seg_attn_forward);
 *            q and lse are overwritten with the host contents first; out
 *            receives the written elements, its other elements are left
 *            unspecified.
 * workspace  as for rk_seg_attn_forward.
 * Asynchronous on `stream`: work queued on `stream` before the call runs
 * first, and `stream` continues only after out_host and lse_host hold the
 * results.  Calls on one plan must not overlap (they share its copy streams
 * and events).  Errors: as rk_seg_attn_forward. */
rk_status_t rk_seg_attn_forward_host(rk_seg_attn_plan_t plan, const void* q_host, void* out_host,
                                     float* lse_host, void* q, void* out, float* lse,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* Stand-alone segment LSE merge (paper, RoPE-orthogonality paragraph).
 * o_parts    device fp32 [P, rows, H, d_v]   partial outputs (normalised)
 * lse_parts  device fp32 [P, rows, H]        partial LSEs; -inf = empty part
 * out        device bf16 [rows, H, d_v]      merged output (round to nearest even)
 * lse_out    device fp32 [rows, H]           lse = ln sum_j exp(lse_j)
 * Parts with lse = -inf carry weight 0; if all are -inf the result is
 * out = 0, lse = -inf.  P >= 1, rows >= 0, 1 <= H, 1 <= d_v <= 1024.
 * Asynchronous on `stream`.  Errors: RK_ERR_NULL, RK_ERR_INVALID_ARG,
 * RK_ERR_ALIGNMENT, RK_ERR_CUDA. */
rk_status_t rk_lse_merge(const float* o_parts, const float* lse_parts, int32_t P,
                         int64_t rows, int32_t H, int32_t d_v, void* out, float* lse_out,
                         void* stream);

/* Size of the device array that rk_seg_attn_forward_noalloc uses as scratch. */
#define RK_NOALLOC_SCRATCH_BYTES (32u << 20)

/* rk_seg_attn_forward for callers that cannot allocate device memory when
 * they issue the forward (engines that reserve all memory up front, code
 * that cannot reach an allocator).  The paper has no counterpart: this is a
 * memory-management variant of rk_seg_attn_forward, with the same
 * arguments minus the workspace and the same results.  The scratch that
 * rk_seg_attn_forward takes as `workspace` lives instead in one file-scope
 * device array of RK_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads
 * the library holds until the process exits.  The call allocates nothing.
 * All calls on a device share that array and it keeps the previous call's
 * contents (each call clears what must start at zero); calls whose kernels
 * overlap on the GPU race on it, so order them on one stream.  The first
 * call on a device looks up the array's address with that device current,
 * and a call that finds a new context on the device (after cudaDeviceReset)
 * looks it up again; make those calls before any stream capture.
 * Errors: as rk_seg_attn_forward, plus RK_ERR_CAPACITY (before any launch)
 * when rk_seg_attn_workspace_bytes(plan) > RK_NOALLOC_SCRATCH_BYTES. */
rk_status_t rk_seg_attn_forward_noalloc(rk_seg_attn_plan_t plan, const void* q, void* out,
                                        float* lse, void* stream);

/* Synchronise `stream`, return and clear the plan's device status word
 * (RK_OK, or RK_ERR_DEVICE_TIMEOUT if a bounded wait expired). */
rk_status_t rk_seg_attn_last_device_status(rk_seg_attn_plan_t plan, void* stream);

/* Static description of a status code (never NULL). */
const char* rk_status_string(rk_status_t status);

/* ---- protected-row set on the device ---------------------------------- */

/* Rule flag: no boundary, Bernoulli or budget rows (only new and dirty rows). */
#define RK_PROT_NONE 1u

/* Device scratch (bytes) rk_protected_build needs for num_requests requests
 * with num_segments segments in total (0 for invalid counts). */
size_t rk_protected_workspace_bytes(int32_t num_requests, int32_t num_segments);

/* Build the protected-row bitmap of every request on the device (paper,
 * protected-set paragraph: the union of query rows, new rows, dirty rows,
 * the first and last rows of every relocated segment and Indexer-selected
 * rows, grown by a fixed controller to a 10 / 20 / 25 % budget).  Per
 * request (segments in the layout of rk_seg_attn_desc_t; the latent
 * pointers are ignored):
 *   - rows of RK_SEG_NEW segments and rows whose `dirty` bit is set are
 *     protected;
 *   - unless RK_PROT_NONE: the first and last `boundary` rows of every
 *     cached segment are protected, and then
 *       p_random > 0:   every cached row with u[row] < p_random (compared in
 *                       double precision);
 *       budget_pct > 0: until ceil(budget_pct * C / 100) of the C cached rows
 *                       are protected (boundary rows first, all of them kept
 *                       if they alone exceed it), the non-boundary cached rows
 *                       with the highest score, ties to the lower row (the
 *                       score vector stands in for the Indexer; finite values;
 *                       -0 ranks as +0).
 * u, score   device arrays, the requests' rows concatenated (T_r entries per
 *            request); u may be NULL unless p_random > 0, score unless
 *            budget_pct > 0.
 * dirty      device uint32 words in the bitmap layout below, or NULL.
 * bitmap     device uint32 out: per request ceil(T_r / 32) words, requests
 *            concatenated; bit p % 32 of word p / 32 set when row p is
 *            protected (LSB first).  Usable as rk_seg_attn_desc_t's bitmap
 *            with RK_PLAN_DEVICE_BITMAP.
 * workspace  device scratch of rk_protected_workspace_bytes bytes, 16-byte
 *            aligned; overwritten.
 * Asynchronous on `stream`.  Errors: RK_ERR_NULL, RK_ERR_INVALID_ARG,
 * RK_ERR_SEGMENT_OVERLAP, RK_ERR_SEGMENT_GAP, RK_ERR_CAPACITY,
 * RK_ERR_WORKSPACE, RK_ERR_ALIGNMENT, RK_ERR_CUDA. */
rk_status_t rk_protected_build(int32_t num_requests, const int32_t* seg_begin,
                               const rk_segment_t* segs, int32_t boundary, double p_random,
                               int32_t budget_pct, uint32_t rule_flags, const double* u,
                               const float* score, const uint32_t* dirty, uint32_t* bitmap,
                               void* workspace, size_t workspace_bytes, void* stream);

/* ---- projected state and layer output ----------------------------------- */

/* Shapes of the projection that follows the attention (paper, first
 * paragraphs: eqs. 2-4; TP8 fast-path paragraph).  Heads act in their native
 * output groups of 8 consecutive heads; each group has its own block of the
 * first output projection W_a. */
typedef struct {
  int64_t rows;              /* computed rows (as the attention's out) */
  int32_t num_heads;         /* H, a multiple of 8, at most 256 */
  int32_t d_v;               /* per-head output width (512) */
  int32_t d_g;               /* projected width per group, a multiple of 256 */
  int32_t d_model;           /* layer output width, a multiple of 256 */
  const uint8_t* head_role;  /* host [H]: 0 Local, 1 Global */
} rk_project_desc_t;

/* Projected state and layer output with row-wise replacement of the Local
 * contribution (paper: sliced W_a projection, Local restoration and row-wise
 * replacement into a contiguous projected state, W_b once; blog: z = z_off +
 * z_on, y = W_b z).  For every row t and group g:
 *   z[t, g] = W_aG(g) O_G[t] + (row t protected ? W_aL(g) O_L[t] : z_off[t, g])
 *   y[t]    = W_b z[t]
 * where W_aG(g) / W_aL(g) are the columns of group g's W_a block that belong
 * to its Global / Local heads.  bf16 operands, fp32 accumulation, bf16
 * results.  The inverse output rotation is the identity (the values carry
 * no rotary part).
 * o         device bf16 [rows, H, d_v]: the attention output (its Local heads
 *           hold fresh values on the protected rows).
 * z_off     device bf16 [rows, H / 8, d_g]: the cached projected Local
 *           contribution of every row.
 * prot      device uint32 [ceil(rows / 32)]: bit r % 32 of word r / 32 set
 *           when row r is protected.
 * w_a       device bf16 [H / 8, d_g, 8 d_v], row-major per group.
 * w_b       device bf16 [d_model, (H / 8) d_g], row-major.
 * z         device bf16 [rows, (H / 8) d_g], out (the projected state).
 * y         device bf16 [rows, d_model], out.
 * status    device int32, 0 on entry; a bounded device wait that expires
 *           stores RK_ERR_DEVICE_TIMEOUT.
 * All device pointers 16-byte aligned (prot and status 4-byte).  Allocates
 * nothing; asynchronous on `stream`.  Errors: RK_ERR_NULL,
 * RK_ERR_INVALID_ARG, RK_ERR_UNSUPPORTED_DIMS (d_v != 512), RK_ERR_ALIGNMENT,
 * RK_ERR_CAPACITY, RK_ERR_CUDA. */
rk_status_t rk_project_forward(const rk_project_desc_t* desc, const void* o, const void* z_off,
                               const uint32_t* prot, const void* w_a, const void* w_b, void* z,
                               void* y, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RK_SEG_ATTN_H */
