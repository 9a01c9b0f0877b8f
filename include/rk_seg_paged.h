/*
 * rk_seg_paged.h - C ABI of SegPagedAttention for grouped-query attention.
 *
 * The operation is the attention prefill of the original RedKnot scheme for
 * GQA models (RedKnot blog "RedKnot, explained", "Insight 3: savings must show
 * up in memory", with the head roles of "Insight 1"):
 *
 *   - the KV cache is stored per KV head in pages; a Global head keeps pages
 *     for the whole prompt, a Local head only the pages of its sink and
 *     window, so no mask over the prompt is needed and every head stays on
 *     the fast path;
 *   - every query head of a KV group attends to the keys of that KV head its
 *     role makes visible: Global heads every k <= p, Local heads k <= p with
 *     k < sink or k >= p - window (blog "Insight 1", the window W(i)).
 *
 * Conventions
 * -----------
 * bf16       IEEE bfloat16 stored as uint16.
 * head_dim   d = 128.  Keys carry their RoPE at absolute positions, unless
 *            their block belongs to a relocated document (block_delta below).
 * pages      k_pages and v_pages are bf16 [num_pages, page_size, d] with
 *            page_size = 128: a page holds 128 consecutive tokens of ONE KV
 *            head.  Logical block b of a sequence covers tokens
 *            [128 b, 128 b + 128).  Rows of a sequence's last page beyond its
 *            length must hold finite values (they meet probability 0).
 * groups     query head i belongs to KV head i / G with G = Hq / Hkv.
 * rows       per request r in order, the absolute positions q_row_begin[r] ..
 *            T_r - 1 are computed; q, out and lse are indexed by this
 *            flattened row index.
 * scores     x = softmax_scale * q.k; lse is the natural-log LSE of x.
 * errors     argument and geometry errors are returned synchronously before
 *            any launch; a failed CUDA call returns RK_ERR_CUDA; a bounded
 *            device wait that expires is reported by
 *            rk_segpaged_last_device_status.  There is no fallback path.
 * Status codes are the rk_status_t values of rk_seg_attn.h.
 */
#ifndef RK_SEG_PAGED_H
#define RK_SEG_PAGED_H

#include <stddef.h>
#include <stdint.h>

#include "rk_seg_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Plan flags. */
#define RK_SEGPAGED_HOST_ONLY 1u   /* build and validate on the host only */
#define RK_SEGPAGED_DENSE_MASK 2u  /* the "dense + mask" arm the blog compares
                                      against: Local heads walk every block of
                                      the prompt and hide what they cannot see
                                      with the element mask (same results,
                                      the work of full causal attention);
                                      needs every block of every KV head */

/* Geometry and roles.  Every pointer is a HOST pointer, read only during
 * rk_segpaged_plan.
 * num_requests   R >= 1.
 * seq_len        [R] T_r >= 1 tokens of request r.
 * q_row_begin    [R] first computed row, 0 <= q_row_begin[r] < T_r (0 for a
 *                prefill, T_r - 1 for a decode step).
 * num_q_heads    Hq; num_kv_heads Hkv; Hq = G Hkv with G in {1, 2, 4, 8, 16}.
 * head_dim       128.
 * page_size      128.
 * num_pages      pages in k_pages and v_pages (>= 1).
 * max_blocks     columns of block_table (>= ceil(max T_r / 128)).
 * block_table    [R][Hkv][max_blocks] physical page of logical block b of KV
 *                head g in request r, or -1 where the head keeps no page.
 *                Every block that a computed row can see must have a page.
 * kv_head_role   [Hkv] 0 = Local, 1 = Global.
 * sink, window   Local visibility: k <= p with k < sink or k >= p - window.
 * softmax_scale  s > 0.
 * flags          RK_SEGPAGED_* bits.
 * block_delta    [R][max_blocks] or NULL.  Relocated documents (RedKnot blog,
 *                "Insight 1": a document cached alone and reused at offset
 *                delta; RedKnot-MLA paper, RoPE-orthogonality paragraph: the
 *                query turns by -delta instead of the cache being rewritten):
 *                the keys of logical block b of request r, in every KV head,
 *                carry their RoPE at position k - block_delta[r][b] instead of
 *                k.  Entries must lie in [-2^31, 2^31).  NULL: every key at its
 *                absolute position.  A plan with offsets runs every tile on the
 *                one-sub-tile kernel, whose query operand is R(-delta) q kept
 *                as bf16 hi + lo parts (rewritten at each change of offset
 *                along the key walk; a zero offset skips the lo part).
 * rope_base      RoPE base of the keys and queries (pairs (2j, 2j + 1) over
 *                all 128 dims, theta_j = base^(-2j/128)); read only with
 *                block_delta. */
typedef struct {
  int32_t num_requests;
  const int64_t* seq_len;
  const int64_t* q_row_begin;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int64_t num_pages;
  int32_t max_blocks;
  const int32_t* block_table;
  const uint8_t* kv_head_role;
  int32_t sink;
  int32_t window;
  float softmax_scale;
  uint32_t flags;
  const int64_t* block_delta;
  double rope_base;
} rk_segpaged_desc_t;

typedef struct rk_segpaged_plan_s* rk_segpaged_plan_t;

/* Host-side counts of a plan. */
typedef struct {
  int64_t rows;             /* computed rows */
  int64_t tiles;            /* work tiles: (request, KV head, 128 / G rows) */
  int64_t pairs;            /* attended (row, query head, key) pairs */
  int64_t performed_pairs;  /* 16, 128 or 256 pairs x 128 keys per issued
                               (tile, key block): decode, one or two
                               sub-tiles */
  int64_t kv_blocks;        /* key blocks read, summed over tiles */
  int64_t split_parts;      /* parts of split tiles (0 if none) */
  int32_t group;            /* G */
  int32_t reserved;
} rk_segpaged_info_t;

/* Validate the descriptor, check that every block a computed row can see has
 * a page (RK_ERR_INVALID_ARG otherwise), list the tiles longest first and
 * upload them with a copy of the block table on `stream`.  A tile with few
 * query pairs in use and a long key walk is split into parts of 32 blocks:
 * at most 16 pairs (a decode step) and more than 48 blocks, or 17 to 64
 * pairs and more than 64 blocks.  The parts'
 * normalised partial outputs and LSEs are merged by log-sum-exp in the
 * workspace by the last part to finish (the RedKnot-MLA paper's numerically
 * stable merge, RoPE-orthogonality paragraph).
 * Errors: RK_ERR_NULL, RK_ERR_INVALID_ARG, RK_ERR_UNSUPPORTED_DIMS (head_dim,
 * page_size or G), RK_ERR_CAPACITY, RK_ERR_CUDA.  On error *out is NULL. */
rk_status_t rk_segpaged_plan(const rk_segpaged_desc_t* desc, void* stream,
                             rk_segpaged_plan_t* out);

/* Attention over the pages (blog "Insight 3").
 * q        device bf16 [rows, Hq, 128], 16-byte aligned.
 * k_pages  device bf16 [num_pages, 128, 128]; v_pages likewise; 16-byte
 *          aligned; owned by the caller.
 * out      device bf16 [rows, Hq, 128], written on every computed row.
 * lse      device fp32 [rows, Hq], written likewise.
 * workspace device scratch of rk_segpaged_workspace_bytes(plan) bytes,
 *          16-byte aligned; contents on entry irrelevant.
 * Asynchronous on `stream`.  Errors: RK_ERR_NULL, RK_ERR_ALIGNMENT,
 * RK_ERR_WORKSPACE, RK_ERR_PLAN_MISMATCH, RK_ERR_CUDA. */
rk_status_t rk_segpaged_forward(rk_segpaged_plan_t plan, const void* q, const void* k_pages,
                                const void* v_pages, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Bytes of device workspace rk_segpaged_forward needs (0 when no tile is
 * split; then workspace may be NULL).  Forwards sharing a workspace must be
 * ordered on one stream. */
size_t rk_segpaged_workspace_bytes(rk_segpaged_plan_t plan);

/* Plan counts.  Errors: RK_ERR_NULL. */
rk_status_t rk_segpaged_plan_info(rk_segpaged_plan_t plan, rk_segpaged_info_t* info);

/* Synchronise `stream`, return RK_ERR_DEVICE_TIMEOUT if a bounded device wait
 * of a forward on this plan expired since the last call (and clear it), else
 * RK_OK. */
rk_status_t rk_segpaged_last_device_status(rk_segpaged_plan_t plan, void* stream);

/* Release a plan (synchronises the device first; NULL is ignored). */
void rk_segpaged_plan_destroy(rk_segpaged_plan_t plan);

#ifdef __cplusplus
}
#endif

#endif /* RK_SEG_PAGED_H */
