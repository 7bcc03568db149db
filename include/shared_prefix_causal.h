/*
 * shared_prefix_causal.h -- C ABI of the shared-prefix tree attention library.
 *
 * Several model calls whose token prefixes match exactly are packed once as a
 * tree of token segments, laid out in DFS preorder with each segment's start,
 * length, parent and depth ("[ENHANCEMENT] Shared-prefix training with context
 * parallelism for exact agent trajectories", issue #7386, "Describe the
 * solution you'd like", first bullet; "TreePackedSeqParams" PR #7387,
 * "Summary", first bullet).  A query token attends causally inside its own
 * segment and fully to every ancestor segment, and to nothing else (issue
 * #7386, third bullet; PR #7387, second bullet).  The result equals packing
 * every root-to-leaf call on its own (issue #7386, "Describe alternatives
 * you've considered", item 1) while each shared prefix's K/V is stored once.
 *
 * General conventions
 *  - Every call returns an int status (sp_status); nothing throws across the
 *    ABI.  A non-zero host return means nothing was launched, except
 *    SP_ERR_CUDA, which reports a failed launch.
 *  - Device pointers are CUDA global-memory pointers that the caller owns and
 *    keeps alive until the work on `stream` has finished; every tensor is
 *    dense (contiguous) in the layout given below and 16-byte aligned
 *    (SP_ERR_ALIGNMENT otherwise).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  All device work is asynchronous on that stream.
 *  - `d_status` (nullable) is a device int32 into which kernels OR the
 *    SP_DEV_* bits of errors they detect while running; the caller zeroes it
 *    before the call and reads it after synchronising.
 *  - Head layout (grouped-query attention): Hq query heads, Hkv key/value
 *    heads, G = Hq / Hkv; query head h reads key/value head h / G.
 *  - The ABI takes no mask, window, bias or soft-cap: unsupported attention
 *    modifiers cannot be requested (issue #7386, sixth bullet; PR #7387,
 *    fifth bullet: reject unsupported modifiers instead of ignoring them).
 */
#ifndef SHARED_PREFIX_CAUSAL_H
#define SHARED_PREFIX_CAUSAL_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SP_API __attribute__((visibility("default")))
#else
#define SP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SP_OK = 0,
  SP_ERR_INVALID_TREE = -1, /* tree metadata is malformed or not in DFS preorder */
  SP_ERR_INVALID_ARG = -2,  /* null pointer, negative size, size mismatch */
  SP_ERR_UNSUPPORTED = -3,  /* dtype / head_dim / GQA ratio / plan tiling not supported */
  SP_ERR_ALIGNMENT = -4,    /* a tensor pointer is not 16-byte aligned */
  SP_ERR_CUDA = -5,         /* a CUDA runtime or driver call failed */
  SP_ERR_TIMEOUT = -6,      /* (device) a bounded wait gave up */
  SP_ERR_INDEX_RANGE = -7,  /* (device) an edge index outside [0, T) */
  SP_ERR_WORKSPACE = -8,    /* workspace missing or smaller than required */
  SP_ERR_NOT_UPLOADED = -9, /* the plan has no device copy (call sp_plan_upload) */
  SP_ERR_CAP = -10          /* a root path is longer than the fragment token cap */
} sp_status;

/* Bits a kernel ORs into *d_status. */
#define SP_DEV_INDEX_RANGE 1 /* edge_gather met an index outside [0, T); that row is zero-filled */
#define SP_DEV_TIMEOUT 2     /* a pipeline wait in an attention kernel exceeded its spin limit */
#define SP_DEV_BAD_PLAN 4    /* a plan entry points outside [0, T); the work item was skipped */
#define SP_DEV_SMEM_LAYOUT 8 /* a CTA's shared memory did not start where its layout needs; it ran nothing */

typedef enum { SP_BF16 = 0, SP_F32 = 1 } sp_dtype;

/* Tree metadata (host pointers, caller-owned, read only during sp_tree_plan).
 * Segment s owns tokens [seg_start[s], seg_start[s] + seg_len[s]); segments
 * are in DFS preorder; parent[s] < s, or -1 for a root (several roots make a
 * forest, e.g. packed GRPO stars, #7914 introduction); depth[s] = 0 at a
 * root, else depth[parent[s]] + 1.  Segments must tile [0, total_tokens)
 * densely and be non-empty.  num_segments == 0 with total_tokens == 0 is the
 * empty tree (a plan with no work). */
typedef struct {
  int32_t num_segments;
  int32_t total_tokens;
  const int32_t *seg_start;
  const int32_t *seg_len;
  const int32_t *parent;
  const int32_t *depth;
} sp_tree_desc;

/* Opaque plan; library-owned (host and device copies) until sp_plan_destroy. */
typedef struct sp_plan sp_plan;

/* Read-only view of a plan's host tables (valid until sp_plan_destroy).
 *   tiles  [n_tiles][5]  = {seg, q_start, q_end, r_begin, r_count}
 *   ranges [n_ranges][2] = {kv_start, kv_end}; tile t reads ranges
 *                          [r_begin, r_begin + r_count); the last one is causal
 *                          (key j visible to query i iff j <= i), the others
 *                          fully visible
 *   bwd    [n_bwd][5]    = {seg, kv_start, kv_end, q_begin, q_end}: the keys
 *                          [kv_start, kv_end) are seen exactly by the queries
 *                          [q_begin, q_end) with j <= i */
typedef struct {
  int32_t tile_tokens, kv_block, order;
  int32_t total_tokens, num_segments;
  int32_t n_tiles, n_ranges, n_bwd, max_ranges_per_tile;
  const int32_t *tiles;
  const int32_t *ranges;
  const int32_t *bwd;
} sp_plan_info;

/* tree_plan -- validate the tree and build the per-query-tile ancestor
 * KV-range lists (issue #7386, "Describe the solution you'd like", third
 * bullet: every query run attends to its own ancestor path and nothing else;
 * PR #7387, "Summary": a query segment attends causally over its ancestors).
 *   tile_tokens  query tokens per tile (> 0); a tile never crosses a segment
 *                end.  The bf16 kernels need tile_tokens * G == 128; the fp32
 *                kernels need tile_tokens * G <= 128.
 *   kv_block     keys per backward block (> 0); bf16 needs 128, fp32 <= 128.
 *   order        0: tiles sorted so that tile k of all siblings run back to back
 *                (shared ancestor K/V stays in L2); 1: longest KV walk first.
 *   *out         receives the new plan (NULL on error).
 * Errors: SP_ERR_INVALID_ARG (null pointers, bad sizes), SP_ERR_INVALID_TREE
 * (checks listed in sp_tree_desc; #7914, introduction: unsupported layouts
 * are refused before anything runs), SP_ERR_UNSUPPORTED (the plan would hold
 * more than 2^30 root-path intervals or tile ranges: its tables are indexed
 * in int32; only very deep trees whose paths do not merge come near this). */
SP_API int sp_tree_plan(const sp_tree_desc *tree, int32_t tile_tokens, int32_t kv_block, int32_t order,
                 sp_plan **out);

/* Fills *info with the plan's host tables.  Errors: SP_ERR_INVALID_ARG. */
SP_API int sp_plan_view(const sp_plan *plan, sp_plan_info *info);

/* The key blocks the bf16 backward runs (host copies, valid until
 * sp_plan_destroy), built with the device tables (first upload or
 * sp_plan_device_bytes; this call builds them too if needed, so it falls
 * under the same rule: one thread makes the first of these calls).  The backward
 * sums every branch's contribution into the prefix the branches share (#7914,
 * introduction), so a block of keys walks the query run that sees them.  A
 * segment's last, partial kv_block of keys is filled with the leading keys of
 * the segments of its subtree that follow it in token order:
 *   *rows     [*n_rows][5] = {seg of the first key, kv_start, kv_end,
 *             q_begin = kv_start, q_end}, in launch order; every key of
 *             [kv_start, kv_end) has q_end >= its own run end
 *   *key_end  [total_tokens]: the end of each key's query run (the subtree end
 *             of its segment); key j is seen by query i iff j <= i < key_end[j]
 * Ownership stays with the plan.  Errors: SP_ERR_INVALID_ARG (null pointers),
 * SP_ERR_UNSUPPORTED (as sp_plan_device_bytes). */
SP_API int sp_plan_bwd_blocks(sp_plan *plan, const int32_t **rows, int32_t *n_rows, const int32_t **key_end);

/* Copies the plan tables to device memory owned by the plan (a cudaMalloc on
 * the current device and an async copy on `stream`).  Must precede the first
 * attention call with this plan; repeat calls are no-ops.  The first upload
 * (this call or sp_plan_upload_to), or sp_plan_device_bytes, builds the device
 * tables inside the plan, so one thread must make those calls; after that the plan is read-only and any number of
 * calls on any streams of that device may use it at once.
 * Errors: SP_ERR_INVALID_ARG, SP_ERR_CUDA, SP_ERR_UNSUPPORTED (the forward's
 * block lists could pass 2^30 entries: the tiles' ranges hold that many 128-key
 * blocks, as a single sequence of a few million tokens cut into small tiles
 * does). */
SP_API int sp_plan_upload(sp_plan *plan, void *stream);

/* Bytes of device memory the plan's tables take (for sp_plan_upload_to);
 * 0 for a NULL plan or one sp_plan_upload would refuse as SP_ERR_UNSUPPORTED. */
SP_API size_t sp_plan_device_bytes(sp_plan *plan);

/* sp_plan_upload into caller-owned device memory: no allocation and no
 * synchronisation.  The tables are copied on `stream` (the host copies are
 * staged before the call returns), so kernels launched on the same stream
 * afterwards see them; the caller keeps the buffer alive, and unmodified,
 * while any kernel using the plan may run, and frees it (sp_plan_destroy
 * does not).  A training loop can plan every step without device
 * allocations.  Repeat calls, or a call after sp_plan_upload, are no-ops.
 *   device_buffer  256-byte aligned, at least sp_plan_device_bytes(plan) bytes.
 * Errors: SP_ERR_INVALID_ARG, SP_ERR_ALIGNMENT, SP_ERR_WORKSPACE (too small),
 * SP_ERR_CUDA, SP_ERR_UNSUPPORTED (as sp_plan_upload). */
SP_API int sp_plan_upload_to(sp_plan *plan, void *device_buffer, size_t buffer_bytes, void *stream);

/* Frees the plan (host copies, and the device copy if sp_plan_upload made
 * it).  NULL is ignored.  The caller must make sure no queued kernel still
 * reads the plan. */
SP_API void sp_plan_destroy(sp_plan *plan);

/* ---------------------------------------------------- bounded fragments
 * A tree too large for one step is split into fragments of at most
 * max_tokens physical tokens.  The trainer keeps every fragment under a memory
 * bound, repeating ancestors in several fragments where it has to, and every
 * sampled action keeps exactly one loss owner (issue #7386, "Describe the solution
 * you'd like", last paragraph; "Additional context": 3,744,651 physical
 * tokens before fragment duplication, 3,919,929 after).  The pages give no
 * algorithm; this one visits segments in preorder and adds each, with the
 * ancestors the current fragment lacks, while the fragment stays within the
 * cap, else it starts the next fragment from the segment's root path.  Every
 * fragment is closed under "parent of" (each segment comes with its whole
 * root path, so its attention is the same as in the whole tree); the fragment
 * that takes a segment in its own visit owns it (its tokens' outputs and
 * loss); re-added ancestors are context only. */
typedef struct sp_fragments sp_fragments;

/* Read-only view of a fragment plan (valid until sp_fragment_destroy).
 * Fragment f consists of entries [offsets[f], offsets[f+1]) in preorder:
 *   seg[i]           the segment in the input tree
 *   owned[i]         1 if fragment f owns that segment, 0 if it is context
 *   local_parent[i]  the parent as an entry index within fragment f (-1: root)
 *   local_start[i]   the segment's first token in fragment f's packed buffer
 * so (local_start, seg_len[seg], local_parent, depth[seg]) is fragment f's
 * own sp_tree_desc; tokens[f] is its length. */
typedef struct {
  int32_t num_fragments, num_entries;
  int64_t physical_tokens;  /* tokens of the input tree */
  int64_t fragment_tokens;  /* sum of tokens[f] (>= physical_tokens; the ratio is the duplication) */
  const int32_t *offsets;   /* [num_fragments + 1] */
  const int32_t *tokens;    /* [num_fragments] */
  const int32_t *seg, *owned, *local_parent, *local_start; /* [num_entries] */
} sp_fragment_info;

/* Plans the fragments of a validated tree with at most max_tokens tokens
 * each (host only).  *out receives a library-owned handle (NULL on error),
 * freed with sp_fragment_destroy; the tree's arrays are only read during the
 * call.  Errors: SP_ERR_INVALID_ARG (null, max_tokens < 1),
 * SP_ERR_INVALID_TREE, SP_ERR_CAP (a root path longer than max_tokens),
 * SP_ERR_UNSUPPORTED (the sum over segments of depth + 1 passes 2^30: the
 * tables, indexed in int32, could overflow). */
SP_API int sp_fragment_plan(const sp_tree_desc *tree, int64_t max_tokens, sp_fragments **out);
/* Fills *info.  Errors: SP_ERR_INVALID_ARG. */
SP_API int sp_fragment_view(const sp_fragments *frag, sp_fragment_info *info);
/* Frees the fragment plan; NULL is ignored. */
SP_API void sp_fragment_destroy(sp_fragments *frag);

/* tree_attn_fwd -- O and LSE of shared-prefix tree attention.  Query token i
 * attends causally inside its own segment and fully to the tokens of every
 * ancestor segment (issue #7386, "Describe the solution you'd like", third
 * bullet; PR #7387, "Summary", second bullet); the prompt's K/V is read once
 * for all its branches and each branch is isolated from its siblings (#7914,
 * introduction).
 *   q   [T][Hq][D], k and v [T][Hkv][D], o [T][Hq][D]: dtype (bf16 or fp32)
 *   lse [Hq][T] fp32: natural-log sum of exp(softmax_scale * q.k) over the
 *       visible keys (the softmax normaliser, kept for the backward pass)
 *   D in {64, 128}; G = Hq / Hkv in {1, 2, 4, 8}; T == plan total_tokens.
 * bf16 runs on the tensor cores (fp32 accumulation and softmax, P rounded to
 * bf16 for the P*V product); fp32 runs a full-fp32 SIMT kernel.
 * The current device must be the one the plan was uploaded on (its tables
 * live there); otherwise SP_ERR_INVALID_ARG and nothing is launched.
 * Errors: SP_ERR_INVALID_ARG, SP_ERR_UNSUPPORTED, SP_ERR_ALIGNMENT,
 * SP_ERR_NOT_UPLOADED, SP_ERR_CUDA; device: SP_DEV_TIMEOUT, SP_DEV_BAD_PLAN. */
SP_API int sp_tree_attn_fwd(const sp_plan *plan, int32_t dtype, const void *q, const void *k,
                     const void *v, void *o, float *lse, int32_t T, int32_t Hq, int32_t Hkv,
                     int32_t D, float softmax_scale, int32_t *d_status, void *stream);

/* Bytes of device workspace sp_tree_attn_bwd needs for these sizes:
 * 4 * T * Hq (Delta), plus 4 * T * Hq * D (the fp32 dQ accumulator) for bf16,
 * each rounded up to 256.  0 for T <= 0 or a non-positive size. */
SP_API size_t sp_tree_attn_bwd_workspace_bytes(int32_t dtype, int32_t T, int32_t Hq, int32_t D);

/* tree_attn_bwd -- dQ, dK, dV of L = sum_i <O_i, dO_i> through the tree
 * attention (FlashAttention-style: S and P are recomputed from q, k and lse).
 * Every child branch's contribution to a shared prefix's dK/dV is summed into
 * that prefix (#7914, introduction: the backward sums the branches'
 * contributions into the prefix they share).
 *   q, k, v, o, lse, d_o: as in / out of tree_attn_fwd (d_o like o)
 *   dq [T][Hq][D], dk and dv [T][Hkv][D]: outputs in dtype, fully overwritten
 *   workspace: device scratch of at least
 *       sp_tree_attn_bwd_workspace_bytes(dtype, T, Hq, D) bytes, caller-owned;
 *       its contents on entry do not matter.
 * Errors: as sp_tree_attn_fwd, plus SP_ERR_WORKSPACE. */
SP_API int sp_tree_attn_bwd(const sp_plan *plan, int32_t dtype, const void *q, const void *k,
                     const void *v, const void *o, const float *lse, const void *d_o, void *dq,
                     void *dk, void *dv, void *workspace, size_t workspace_bytes, int32_t T,
                     int32_t Hq, int32_t Hkv, int32_t D, float softmax_scale, int32_t *d_status,
                     void *stream);

/* Bytes of device workspace sp_edge_gather_bwd needs (per-token counts and
 * offsets, one int per edge).  0 for a negative size. */
SP_API size_t sp_edge_gather_bwd_workspace_bytes(int32_t T, int32_t E);

/* edge_gather backward -- grad_hidden[t][:] = sum of grad_out[e][:] over the
 * edges e with idx[e] == t, zero for tokens that are no edge's source.  Each
 * sampled action's gradient flows back to its source token's hidden state;
 * a branch-point token shared by several actions receives their sum (one loss
 * owner per action: issue #7386, "Describe the solution you'd like", fifth
 * bullet).  Sums run in ascending e with fp32 accumulation, so results are
 * identical from run to run.
 *   grad_out [E][hidden_dim], grad_hidden [T][hidden_dim] in dtype (fully
 *   overwritten); idx [E] int32 (device); hidden_dim a multiple of 8;
 *   workspace: at least sp_edge_gather_bwd_workspace_bytes(T, E) bytes.
 * An index outside [0, T) sets SP_DEV_INDEX_RANGE and its row is dropped.
 * Errors: SP_ERR_INVALID_ARG, SP_ERR_UNSUPPORTED, SP_ERR_ALIGNMENT,
 * SP_ERR_WORKSPACE, SP_ERR_CUDA. */
SP_API int sp_edge_gather_bwd(int32_t dtype, const void *grad_out, int32_t E, int32_t hidden_dim,
                              const int32_t *idx, int32_t T, void *grad_hidden, void *workspace,
                              size_t workspace_bytes, int32_t *d_status, void *stream);

/* Bytes of device workspace sp_edge_logprob needs: 8 * E * ceil(V / 256)
 * (per-tile row maxima and sums) + 4 * E (label logits), each 256-aligned.
 * 0 for E < 0 or V < 1. */
SP_API size_t sp_edge_logprob_workspace_bytes(int32_t E, int32_t V);

/* Vocabulary head over the sampled-edge states -- the log-probability that
 * each sampled action assigns to its own token.  Only sampled-edge source
 * states go through the projection, and each action owns exactly one loss
 * term (issue #7386, "Describe the solution you'd like", fifth bullet;
 * PR #7387, "Summary", fourth bullet).  For e in [0, E):
 *     logits[e][v] = sum_d hidden_sel[e][d] * weight[v][d]   (fp32 accumulation)
 *     lse[e]       = log sum_v exp(logits[e][v])
 *     logprob[e]   = logits[e][labels[e]] - lse[e]
 * The [E][V] logits are never written to memory.
 *   dtype: SP_BF16 only.  hidden_sel [E][Hd] (e.g. sp_edge_gather's output)
 *   and weight [V][Hd] (a linear layer's weight layout), row-major, 16-byte
 *   aligned, Hd a multiple of 8; labels [E] int32 (device); logprob, lse [E]
 *   fp32 (device, caller-owned, fully overwritten); workspace at least
 *   sp_edge_logprob_workspace_bytes(E, V) bytes, 256-byte aligned.
 * A label outside [0, V) sets SP_DEV_INDEX_RANGE and yields NaN for that
 * action.  Errors: SP_ERR_INVALID_ARG, SP_ERR_UNSUPPORTED (dtype, Hd),
 * SP_ERR_ALIGNMENT, SP_ERR_WORKSPACE, SP_ERR_CUDA. */
SP_API int sp_edge_logprob(int32_t dtype, const void *hidden_sel, int32_t E, int32_t Hd, const void *weight,
                           int32_t V, const int32_t *labels, float *logprob, float *lse, void *workspace,
                           size_t workspace_bytes, int32_t *d_status, void *stream);

/* Bytes of device workspace sp_edge_logprob_bwd needs: 2 * E * V (bf16
 * dlogits).  0 for E < 0 or V < 1. */
SP_API size_t sp_edge_logprob_bwd_workspace_bytes(int32_t E, int32_t V);

/* Backward of sp_edge_logprob for upstream gradients grad_logprob[e] =
 * dL/dlogprob[e] (each sampled action's single loss term, issue #7386,
 * "Describe the solution you'd like", fifth bullet; the projection backward
 * that PR #7387 "Validation And Known Limitations" reports as passing):
 *     dlogits[e][v]    = grad_logprob[e] * (1[v == labels[e]] - exp(logits[e][v] - lse[e]))
 *     d_hidden_sel[e]  = sum_v dlogits[e][v] * weight[v]          [E][Hd] fp32
 *     d_weight[v]      = sum_e dlogits[e][v] * hidden_sel[e]      [V][Hd] fp32
 * The logits are recomputed; dlogits is rounded to bf16 in the workspace and
 * both products accumulate in fp32.  Outputs are overwritten; pass NULL for
 * one to skip it.  lse is sp_edge_logprob's output.  Requirements as for
 * sp_edge_logprob, plus V a multiple of 8 and a workspace of at least
 * sp_edge_logprob_bwd_workspace_bytes(E, V) bytes, 256-byte aligned; feed
 * d_hidden_sel to sp_edge_gather_bwd (dtype SP_F32) for the hidden-state
 * gradient.  A label outside [0, V) sets SP_DEV_INDEX_RANGE (no one-hot term).
 * Errors: SP_ERR_INVALID_ARG, SP_ERR_UNSUPPORTED, SP_ERR_ALIGNMENT,
 * SP_ERR_WORKSPACE, SP_ERR_CUDA. */
SP_API int sp_edge_logprob_bwd(int32_t dtype, const void *hidden_sel, int32_t E, int32_t Hd, const void *weight,
                               int32_t V, const int32_t *labels, const float *lse, const float *grad_logprob,
                               float *d_hidden_sel, float *d_weight, void *workspace, size_t workspace_bytes,
                               int32_t *d_status, void *stream);

/* sp_tree_attn_bwd with a deterministic dQ: same arguments, workspace and
 * errors.  Instead of adding every key block's dQ partial into an fp32 buffer
 * with atomics (whose order, and so rounding, varies from run to run), each
 * query tile walks its own ancestor key ranges and accumulates dQ in a fixed
 * order (the per-run gradient accumulation of "[ENHANCEMENT] Shared-prefix
 * training ...", issue #7386, "Describe the solution you'd like", made
 * reproducible); dK and dV come from a key-block kernel that takes 128 query
 * rows per step.  dQ, dK and dV are identical bit for bit on every call with
 * the same inputs, and agree with sp_tree_attn_bwd's to within bf16 rounding
 * (the same terms summed in another order).  Recomputes S and dP once more per
 * (query tile, key block) than the default path.  Besides sp_tree_attn_bwd's
 * device codes it may set SP_DEV_SMEM_LAYOUT (the key-block kernel found its
 * shared memory not 1024-byte aligned and ran nothing; dK and dV are then not
 * written). */
SP_API int sp_tree_attn_bwd_deterministic(const sp_plan *plan, int32_t dtype, const void *q, const void *k,
                                          const void *v, const void *o, const float *lse, const void *d_o, void *dq,
                                          void *dk, void *dv, void *workspace, size_t workspace_bytes, int32_t T,
                                          int32_t Hq, int32_t Hkv, int32_t D, float softmax_scale,
                                          int32_t *d_status, void *stream);

/* sp_tree_attn_bwd (deterministic == 0) or sp_tree_attn_bwd_deterministic
 * (deterministic == 1) with a measurement hook; the pages have no counterpart.
 * ev_main_begin and ev_main_end are caller-created cudaEvent_t handles (either
 * may be NULL), recorded on `stream` just before and just after the launch of
 * the backward's main kernel (the per-key-block kernel that forms dK, dV and,
 * in the default mode, the dQ partials), so that the caller can time that
 * kernel alone with cudaEventElapsedTime while the preprocess and dQ kernels
 * run outside the pair.  Results, arguments and errors are otherwise those of
 * the two calls above; the fp32 path has no single main kernel and returns
 * SP_ERR_UNSUPPORTED when an event is given.  The events stay owned by the
 * caller. */
SP_API int sp_tree_attn_bwd_timed(const sp_plan *plan, int32_t dtype, const void *q, const void *k, const void *v,
                                  const void *o, const float *lse, const void *d_o, void *dq, void *dk, void *dv,
                                  void *workspace, size_t workspace_bytes, int32_t T, int32_t Hq, int32_t Hkv,
                                  int32_t D, float softmax_scale, int32_t deterministic, void *ev_main_begin,
                                  void *ev_main_end, int32_t *d_status, void *stream);

/* tree_attn_fwd on pairs of SMs: the same outputs as sp_tree_attn_fwd (to
 * within bf16 rounding of P and O, summed in the same order per tile), from
 * tcgen05 products that span the two SMs of a cluster (cta_group::2): each
 * M = 256 product takes 128 query rows from each SM, and each SM loads half of
 * every K and V block.  The pages name no such kernel; it is a variant of the
 * forward's main kernel, kept beside it because on these workloads it runs
 * slower than the one-SM kernel (the softmax of each tile waits on products
 * and barriers that now cross two SMs).  bf16, head_dim 128 and the tiling of
 * sp_tree_attn_fwd only; other cases return SP_ERR_UNSUPPORTED.  Arguments,
 * layouts and errors as sp_tree_attn_fwd. */
SP_API int sp_tree_attn_fwd_paired(const sp_plan *plan, int32_t dtype, const void *q, const void *k, const void *v,
                                   void *o, float *lse, int32_t T, int32_t Hq, int32_t Hkv, int32_t D,
                                   float softmax_scale, int32_t *d_status, void *stream);

/* Size of the fixed device scratch behind sp_tree_attn_bwd_noalloc (64 MiB). */
#define SP_NOALLOC_SCRATCH_BYTES (64u << 20)

/* tree_attn_bwd without a workspace argument, for callers that cannot
 * allocate device memory (for example code running under a memory pool that
 * owns the whole device, or a plugin that is handed only its inputs and
 * outputs).  The pages have no counterpart: this is a packaging variant of
 * tree_attn_bwd with identical arguments and results, minus the workspace.
 *   Scratch: a fixed SP_NOALLOC_SCRATCH_BYTES array that belongs to the
 *   library's device code, held on every GPU where that code is loaded until
 *   process exit.  The call itself allocates nothing (no cudaMalloc, no
 *   cudaFree, no allocating library routine), but the driver commits the
 *   array's 64 MiB when it loads the library's device code on a device: with
 *   CUDA's default lazy module loading that happens during the first call of
 *   this function on that device; with CUDA_MODULE_LOADING=EAGER, when the
 *   library's device code is loaded into the context.  So make a first call
 *   (or use EAGER loading) before a memory pool takes the whole device, and
 *   before any stream capture: that first call also looks up the array's
 *   device address.  The address is cached per device and context; a new
 *   context (after cudaDeviceReset) is detected and looked up again.  All
 *   calls on a device share the array, so calls that overlap on the GPU race;
 *   serialise them.  Each call rewrites every scratch byte it reads.
 *   Limit: sp_tree_attn_bwd_workspace_bytes(dtype, T, Hq, D) must not exceed
 *   SP_NOALLOC_SCRATCH_BYTES (bf16 needs 4 * T * Hq * (D + 1) bytes, e.g.
 *   T * Hq <= 129,000 rows at D = 128), otherwise SP_ERR_WORKSPACE.
 * Errors: as sp_tree_attn_bwd. */
SP_API int sp_tree_attn_bwd_noalloc(const sp_plan *plan, int32_t dtype, const void *q, const void *k,
                                    const void *v, const void *o, const float *lse, const void *d_o,
                                    void *dq, void *dk, void *dv, int32_t T, int32_t Hq, int32_t Hkv,
                                    int32_t D, float softmax_scale, int32_t *d_status, void *stream);

/* edge_gather -- out[e][:] = hidden[idx[e]][:] for e < E: the sampled-edge
 * source rows that go on to the vocabulary projection (issue #7386, fifth
 * bullet; PR #7387, "Summary", fourth bullet).  hidden [T][hidden_dim] and
 * out [E][hidden_dim] in dtype; idx [E] int32 on the device.  Duplicate
 * indices are legal (one row per sampled action).  hidden_dim * element size
 * must be a multiple of 16 bytes.  An index outside [0, T) zero-fills its
 * row and sets SP_DEV_INDEX_RANGE.  E == 0 is a no-op.
 * Errors: SP_ERR_INVALID_ARG, SP_ERR_UNSUPPORTED, SP_ERR_ALIGNMENT, SP_ERR_CUDA. */
SP_API int sp_edge_gather(int32_t dtype, const void *hidden, int32_t T, int32_t hidden_dim,
                   const int32_t *idx, int32_t E, void *out, int32_t *d_status, void *stream);

/* Diagnostic for failure-detection tests (the pages have no counterpart):
 * launches one warp that waits, with the attention kernels' bounded wait, on
 * an mbarrier nothing ever arrives at.  After spin_limit (>= 256) polls the
 * wait gives up and ORs SP_DEV_TIMEOUT into *d_status (device int32, required).
 * Nothing hangs and the CUDA context stays usable.
 * Errors: SP_ERR_INVALID_ARG, SP_ERR_CUDA. */
SP_API int sp_debug_wait_timeout(int32_t spin_limit, int32_t *d_status, void *stream);

/* Measurement hook for the tail of a launch (the pages have no counterpart).
 * After this call, every launch of the chosen tensor-core kernel records, per
 * CTA b < max_ctas, four uint64 words at device_buffer[4 b]: the global timer
 * (ns) when the CTA started and when it finished, the SM it ran on, and 0.
 * kernel: 1 the forward's main kernel, 2 the backward's per-key-block kernel
 * (either mode), 3 the deterministic backward's per-query-tile dQ kernel; 0 or
 * a NULL buffer turns recording off.  The buffer (16-byte aligned, at least
 * 32 * max_ctas bytes) stays owned by the caller and must outlive the launches;
 * CTAs at or past max_ctas record nothing.  Process-wide setting, read when a
 * kernel is launched; not for use while other threads launch these kernels.
 * Errors: SP_ERR_INVALID_ARG, SP_ERR_ALIGNMENT. */
SP_API int sp_debug_cta_clock(int32_t kernel, void *device_buffer, int64_t max_ctas);

/* Static English text for a status code (never NULL). */
SP_API const char *sp_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SHARED_PREFIX_CAUSAL_H */
