// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "../../include/shared_prefix_causal.h"

struct sp_plan {
  int32_t tile_tokens = 0, kv_block = 0, order = 0;
  int32_t total_tokens = 0, num_segments = 0;
  int32_t max_ranges_per_tile = 0;
  std::vector<int32_t> tiles;   // [n][5]
  std::vector<int32_t> ranges;  // [m][2]
  std::vector<int32_t> bwd;     // [k][5]
  // forward work items derived from the tiles (built at upload): pairs of
  // consecutive tiles and, per pair, the merged list of 128-key blocks
  // runs of 128-key blocks [r][8] = {kb, nb, end[4] (0: not read), causal bits, 0}
  std::vector<int32_t> pairs;   // [p][4] = {tile_a, tile_b or -1, run_begin, run_count}
  std::vector<int32_t> pblk;    // runs of the pairs (slots 0, 1)
  // paired-SM forward work items (built at upload): four tiles per CTA pair
  // and their merged block runs (see build_quads)
  std::vector<int32_t> quads;   // [q][6] = {a0, a1, b0, b1 (or -1), run_begin, run_count}
  std::vector<int32_t> qblk;    // runs of the quads (slots a0, a1, b0, b1)
  // backward key blocks in launch order (built at upload; same rows as bwd),
  // and the total and longest query-run length over them
  std::vector<int32_t> bwd_sched;  // [k][5]
  int64_t bwd_run_sum = 0;
  int32_t bwd_run_max = 0;
  // key blocks of the tensor-core backward (built at upload; see
  // build_bwd_merged), in the same launch order, their runs' sum and maximum,
  // and every key's own query-run end [total_tokens]
  std::vector<int32_t> bwd_merged;  // [m][5]
  int64_t bwdm_run_sum = 0;
  int32_t bwdm_run_max = 0;
  std::vector<int32_t> key_end;
  // device copies (owned), valid after sp_plan_upload
  int32_t *d_tiles = nullptr, *d_ranges = nullptr, *d_bwd = nullptr, *d_pairs = nullptr, *d_pblk = nullptr,
          *d_quads = nullptr, *d_qblk = nullptr, *d_bwdm = nullptr, *d_key_end = nullptr;
  int device = -1;
  bool owns_device = false;  // the device tables were allocated by sp_plan_upload
  int32_t n_tiles() const { return int32_t(tiles.size() / 5); }
  int32_t n_ranges() const { return int32_t(ranges.size() / 2); }
  int32_t n_bwd() const { return int32_t(bwd.size() / 5); }
  int32_t n_pairs() const { return int32_t(pairs.size() / 4); }
  int32_t n_quads() const { return int32_t(quads.size() / 6); }
  int32_t n_bwdm() const { return int32_t(bwd_merged.size() / 5); }
};

namespace spc {

// Tree checks of sp_tree_desc (plan.cpp): SP_OK or SP_ERR_INVALID_TREE.
// Expects num_segments >= 0 and non-null arrays when num_segments > 0.
int validate_tree(const sp_tree_desc &tree);
// Plan builder (plan.cpp).  Returns SP_OK or SP_ERR_INVALID_TREE/ARG.
int build_plan(const sp_tree_desc &tree, int32_t tile_tokens, int32_t kv_block, int32_t order,
               sp_plan &plan);
// Backward launch order (see sp_plan::bwd_sched): rows grouped by the end of
// their query run, latest first, longest run first within a group; also
// builds the merged key blocks (build_bwd_merged).
void build_bwd_schedule(sp_plan &plan);
// The tensor-core backward's key blocks (sp_plan::bwd_merged, key_end): a
// segment's partial last block filled with the leading keys of the segments
// of its subtree that follow it.
void build_bwd_merged(sp_plan &plan);
// Forward pairs and merged block lists from the tiles (see sp_plan::pairs).
void build_pairs(sp_plan &plan, int32_t block_keys);
// Paired-SM forward quads and their merged block lists (see sp_plan::quads).
void build_quads(sp_plan &plan, int32_t block_keys);
// One range of a tile as a run of blocks kb, kb + B, ... (nb of them), all
// ending at the range end; the tile's last range (its own segment) is causal.
struct TileRun {
  int32_t kb, nb, end;
  bool causal;
};
// Merges up to four tiles' run lists by block start into entries of 8 int32
// {kb, nb, end[4], causal bits, 0} appended to runs (see plan.cpp); returns
// the number of entries.
int32_t merge_runs(std::vector<TileRun> (&lists)[4], int32_t block_keys, std::vector<int32_t> &runs);

// Device-side view of a plan passed to kernels by value.
struct PlanDev {
  const int32_t *tiles;
  const int32_t *ranges;
  const int32_t *bwd;
  int32_t n_tiles, n_bwd, tile_tokens, kv_block;
  const int32_t *pairs;
  const int32_t *pblk;
  int32_t n_pairs;
  int64_t bwd_run_sum;  // sum of q1 - q0 over the bwd rows
  int32_t bwd_run_max;  // longest q1 - q0
  const int32_t *quads;
  const int32_t *qblk;
  int32_t n_quads;
  // the tensor-core backward's merged key blocks [n_bwdm][5] (launch order),
  // their runs' sum and maximum, and every key's query-run end [T]
  const int32_t *bwdm;
  int32_t n_bwdm;
  int64_t bwdm_run_sum;
  int32_t bwdm_run_max;
  const int32_t *key_end;
};

// Kernels whose CTAs can record their start and end times (sp_debug_cta_clock).
enum ClockedKernel : int32_t { kClockForward = 1, kClockKeyBlocks = 2, kClockQueryTiles = 3 };
struct CtaClock;
// The record buffer for launches of `kernel` (null buffer when not enabled).
void cta_clock_for(int32_t kernel, unsigned long long **buf, int32_t *cap);

struct AttnShape {
  int32_t T, Hq, Hkv, D, G;
  float scale;
};

// SIMT kernels (attn_simt.cu): any tiling, fp32 arithmetic, input in fp32 or bf16.
int simt_fwd(const PlanDev &p, const AttnShape &s, int32_t dtype, const void *q, const void *k,
             const void *v, void *o, float *lse, int32_t *d_status, void *stream);
int simt_bwd(const PlanDev &p, const AttnShape &s, int32_t dtype, const void *q, const void *k,
             const void *v, const void *o, const float *lse, const void *d_o, void *dq, void *dk,
             void *dv, float *delta, int32_t *d_status, void *stream);

// Tensor-core kernels (sm_103a): bf16 input, tile_tokens * G == 128, kv_block == 128.
int tc_fwd(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, void *o, float *lse,
           int32_t *d_status, void *stream);
// The same forward on a pair of SMs (attn_fwd_pair_sm103a.cu): head_dim 128
// only; SP_ERR_UNSUPPORTED (nothing launched) where it does not apply.
int tc_fwd_pair(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, void *o,
                float *lse, int32_t *d_status, void *stream);
// delta: [Hq][T] fp32 scratch; dqacc: [T][Hq][D] fp32 scratch (zeroed inside;
// unused when deterministic, which computes dQ per query tile with tc_dq).
// ev_begin / ev_end (cudaEvent_t, optional): recorded on the stream just before
// and just after the main kernel's launch, so a caller can time it alone.
int tc_bwd(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, const void *o,
           const float *lse, const void *d_o, void *dq, void *dk, void *dv, float *delta, float *dqacc,
           bool deterministic, int32_t *d_status, void *stream, void *ev_begin = nullptr, void *ev_end = nullptr);
// The default backward's companion passes (attn_bwd_pre_sm103a.cu): Delta =
// rowsum(dO * O) into delta [Hq][T], and zeroing dqacc [T][Hq][D] unless it
// is null; then dq = bf16(scale * dqacc) over n = T * Hq * D values (n % 8 == 0).
int bwd_pre(const AttnShape &s, const void *o, const void *d_o, float *delta, float *dqacc, int sms,
            void *stream);
int dq_convert(const float *dqacc, void *dq, float scale, long n, int sms, void *stream);
// dK and dV only, 128 query rows per step (attn_bwd_kv_sm103a.cu), for the
// deterministic backward; events as tc_bwd.
int tc_bwd_kv(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, const float *lse,
              const void *d_o, void *dk, void *dv, const float *delta, int head_chunk, int32_t *d_status,
              void *stream, void *ev_begin, void *ev_end);
// dQ of every query tile over its own key blocks, no atomics (attn_dq_sm103a.cu);
// delta from the backward's preprocess.
int tc_dq(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, const float *lse,
          const void *d_o, void *dq, const float *delta, int32_t *d_status, void *stream);

// edge_gather and its backward (edge_gather.cu).
// Vocabulary head (lm_head_sm103a.cu): per-action log-probability of the
// sampled label through the projection h W^T, bf16 inputs, fp32 outputs.
size_t lmh_workspace(int32_t E, int32_t V);
int lmh_fwd(const void *hidden_sel, int32_t E, int32_t Hd, const void *weight, int32_t V, const int32_t *labels,
            float *logprob, float *lse, void *workspace, int32_t *d_status, void *stream);
// Backward: bf16 dlogits [E][V] in the workspace, then fp32 d_hidden_sel
// [E][Hd] and d_weight [V][Hd] (either may be null).  V % 8 == 0.
size_t lmh_bwd_workspace(int32_t E, int32_t V);
int lmh_bwd(const void *hidden_sel, int32_t E, int32_t Hd, const void *weight, int32_t V, const int32_t *labels,
            const float *lse, const float *grad_logprob, float *d_hidden_sel, float *d_weight, void *workspace,
            int32_t *d_status, void *stream);
size_t edge_gather_bwd_workspace(int32_t T, int32_t E);
int edge_gather_bwd(int32_t elem_bytes, const void *grad_out, int32_t E, int32_t hidden_dim, const int32_t *idx,
                    int32_t T, void *grad_hidden, void *workspace, int32_t *d_status, void *stream);
int edge_gather(int32_t elem_bytes, const void *hidden, int32_t T, int32_t hidden_dim,
                const int32_t *idx, int32_t E, void *out, int32_t *d_status, void *stream);

}  // namespace spc
