// The C ABI: argument checks, plan ownership and kernel dispatch.  Every
// entry point returns an sp_status and never throws.
#include <cuda_runtime.h>

#include <cstdint>
#include <new>

#include "internal.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_heads(int32_t dtype, int32_t T, int32_t Hq, int32_t Hkv, int32_t D) {
  if (T < 0 || Hq <= 0 || Hkv <= 0) return SP_ERR_INVALID_ARG;
  if (dtype != SP_BF16 && dtype != SP_F32) return SP_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return SP_ERR_UNSUPPORTED;
  if (Hq % Hkv) return SP_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return SP_ERR_UNSUPPORTED;
  return SP_OK;
}

// Tiling each kernel family accepts (see the header's sp_tree_plan notes):
// the tensor-core kernels (bf16) need 128-row query tiles and 128-key blocks;
// the fp32 kernels take any tiling up to those sizes.
int check_tiling(const sp_plan &p, int32_t dtype, int32_t G) {
  if (dtype == SP_BF16) return (p.tile_tokens * G == 128 && p.kv_block == 128) ? SP_OK : SP_ERR_UNSUPPORTED;
  if (p.tile_tokens * G > 128 || p.kv_block > 128) return SP_ERR_UNSUPPORTED;
  return SP_OK;
}

spc::PlanDev plan_dev(const sp_plan &p) {
  return {p.d_tiles, p.d_ranges, p.d_bwd, p.n_tiles(), p.n_bwd(), p.tile_tokens, p.kv_block,
          p.d_pairs, p.d_pblk, p.n_pairs(), p.bwd_run_sum, p.bwd_run_max, p.d_quads, p.d_qblk, p.n_quads(),
          p.d_bwdm, p.n_bwdm(), p.bwdm_run_sum, p.bwdm_run_max, p.d_key_end};
}

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

// A plan's device tables live on the GPU that was current when it was uploaded;
// kernels launched on another GPU must not read them.
bool on_plan_device(const sp_plan &p) {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess && dev == p.device;
}

int32_t g_clock_kernel = 0;
unsigned long long *g_clock_buf = nullptr;
int32_t g_clock_cap = 0;

}  // namespace

namespace spc {
void cta_clock_for(int32_t kernel, unsigned long long **buf, int32_t *cap) {
  const bool on = kernel == g_clock_kernel && g_clock_buf;
  *buf = on ? g_clock_buf : nullptr;
  *cap = on ? g_clock_cap : 0;
}
}  // namespace spc

extern "C" {

int sp_debug_cta_clock(int32_t kernel, void *device_buffer, int64_t max_ctas) {
  if (kernel == 0 || !device_buffer) {
    g_clock_kernel = 0, g_clock_buf = nullptr, g_clock_cap = 0;
    return SP_OK;
  }
  if (kernel < 1 || kernel > 3 || max_ctas <= 0 || max_ctas > (int64_t(1) << 30)) return SP_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(device_buffer) & 15u) return SP_ERR_ALIGNMENT;
  g_clock_kernel = kernel;
  g_clock_buf = static_cast<unsigned long long *>(device_buffer);
  g_clock_cap = int32_t(max_ctas);
  return SP_OK;
}

int sp_tree_plan(const sp_tree_desc *tree, int32_t tile_tokens, int32_t kv_block, int32_t order, sp_plan **out) {
  if (!out) return SP_ERR_INVALID_ARG;
  *out = nullptr;
  if (!tree) return SP_ERR_INVALID_ARG;
  sp_plan *p = new (std::nothrow) sp_plan();
  if (!p) return SP_ERR_INVALID_ARG;
  int rc;
  try {
    rc = spc::build_plan(*tree, tile_tokens, kv_block, order, *p);
  } catch (...) {
    rc = SP_ERR_INVALID_ARG;
  }
  if (rc != SP_OK) {
    delete p;
    return rc;
  }
  *out = p;
  return SP_OK;
}

int sp_plan_view(const sp_plan *p, sp_plan_info *info) {
  if (!p || !info) return SP_ERR_INVALID_ARG;
  info->tile_tokens = p->tile_tokens;
  info->kv_block = p->kv_block;
  info->order = p->order;
  info->total_tokens = p->total_tokens;
  info->num_segments = p->num_segments;
  info->n_tiles = p->n_tiles();
  info->n_ranges = p->n_ranges();
  info->n_bwd = p->n_bwd();
  info->max_ranges_per_tile = p->max_ranges_per_tile;
  info->tiles = p->tiles.data();
  info->ranges = p->ranges.data();
  info->bwd = p->bwd.data();
  return SP_OK;
}

}  // extern "C"

namespace {

// Derived device tables (forward pairs, backward launch order), built once.
int prepare_device_tables(sp_plan *p) {
  if (!p->pairs.empty() || p->tiles.empty()) return SP_OK;
  // The forward's merged lists hold at most one entry per 128-key block of each
  // tile's ranges, indexed in int32: plans that could pass 2^30 are refused.
  int64_t blocks = 0;
  for (size_t r = 0; r + 1 < p->ranges.size(); r += 2) blocks += (int64_t(p->ranges[r + 1]) - p->ranges[r] + 127) / 128;
  if (blocks > (int64_t(1) << 30)) return SP_ERR_UNSUPPORTED;
  try {
    spc::build_pairs(*p, 128);
    spc::build_quads(*p, 128);
    spc::build_bwd_schedule(*p);
  } catch (...) {
    return SP_ERR_INVALID_ARG;
  }
  return SP_OK;
}

struct DeviceLayout {
  size_t bt, br, bb, bp, bk, bq, bqk, bm, be, total;
};

DeviceLayout device_layout(const sp_plan &p) {
  DeviceLayout l{p.tiles.size() * 4, p.ranges.size() * 4, p.bwd.size() * 4,        p.pairs.size() * 4,
                 p.pblk.size() * 4,  p.quads.size() * 4,  p.qblk.size() * 4,       p.bwd_merged.size() * 4,
                 p.key_end.size() * 4, 0};
  l.total = align_up(l.bt) + align_up(l.br) + align_up(l.bb) + align_up(l.bp) + align_up(l.bk) + align_up(l.bq) +
            align_up(l.bqk) + align_up(l.bm) + align_up(l.be) + 256;
  return l;
}

// Copies the tables into base (256-byte aligned) on stream st and points the plan at them.
int copy_tables(sp_plan *p, char *base, const DeviceLayout &l, cudaStream_t st) {
  int32_t *dt = reinterpret_cast<int32_t *>(base);
  int32_t *dr = reinterpret_cast<int32_t *>(base + align_up(l.bt));
  int32_t *db = reinterpret_cast<int32_t *>(base + align_up(l.bt) + align_up(l.br));
  int32_t *dp = reinterpret_cast<int32_t *>(base + align_up(l.bt) + align_up(l.br) + align_up(l.bb));
  int32_t *dk = reinterpret_cast<int32_t *>(base + align_up(l.bt) + align_up(l.br) + align_up(l.bb) + align_up(l.bp));
  int32_t *dq = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(dk) + align_up(l.bk));
  int32_t *dqk = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(dq) + align_up(l.bq));
  int32_t *dm = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(dqk) + align_up(l.bqk));
  int32_t *de = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(dm) + align_up(l.bm));
  if ((l.bt && cudaMemcpyAsync(dt, p->tiles.data(), l.bt, cudaMemcpyHostToDevice, st) != cudaSuccess) ||
      (l.bq && cudaMemcpyAsync(dq, p->quads.data(), l.bq, cudaMemcpyHostToDevice, st) != cudaSuccess) ||
      (l.bqk && cudaMemcpyAsync(dqk, p->qblk.data(), l.bqk, cudaMemcpyHostToDevice, st) != cudaSuccess) ||
      (l.br && cudaMemcpyAsync(dr, p->ranges.data(), l.br, cudaMemcpyHostToDevice, st) != cudaSuccess) ||
      (l.bb && cudaMemcpyAsync(db, p->bwd_sched.data(), l.bb, cudaMemcpyHostToDevice, st) != cudaSuccess) ||
      (l.bp && cudaMemcpyAsync(dp, p->pairs.data(), l.bp, cudaMemcpyHostToDevice, st) != cudaSuccess) ||
      (l.bk && cudaMemcpyAsync(dk, p->pblk.data(), l.bk, cudaMemcpyHostToDevice, st) != cudaSuccess) ||
      (l.bm && cudaMemcpyAsync(dm, p->bwd_merged.data(), l.bm, cudaMemcpyHostToDevice, st) != cudaSuccess) ||
      (l.be && cudaMemcpyAsync(de, p->key_end.data(), l.be, cudaMemcpyHostToDevice, st) != cudaSuccess))
    return SP_ERR_CUDA;
  p->d_tiles = dt;
  p->d_ranges = dr;
  p->d_bwd = db;
  p->d_pairs = dp;
  p->d_pblk = dk;
  p->d_quads = l.bq ? dq : nullptr;
  p->d_qblk = l.bqk ? dqk : nullptr;
  p->d_bwdm = l.bm ? dm : nullptr;
  p->d_key_end = l.be ? de : nullptr;
  cudaGetDevice(&p->device);
  return SP_OK;
}

}  // namespace

extern "C" {

int sp_plan_upload(sp_plan *p, void *stream) {
  if (!p) return SP_ERR_INVALID_ARG;
  if (p->d_tiles) return SP_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (int rc = prepare_device_tables(p)) return rc;
  const DeviceLayout l = device_layout(*p);
  char *base = nullptr;
  if (cudaMalloc(&base, l.total) != cudaSuccess) return SP_ERR_CUDA;
  if (copy_tables(p, base, l, st) != SP_OK || cudaStreamSynchronize(st) != cudaSuccess) {
    p->d_tiles = p->d_ranges = p->d_bwd = p->d_pairs = p->d_pblk = p->d_quads = p->d_qblk = p->d_bwdm =
        p->d_key_end = nullptr;
    cudaFree(base);
    return SP_ERR_CUDA;
  }
  p->owns_device = true;
  return SP_OK;
}

size_t sp_plan_device_bytes(sp_plan *p) {
  if (!p || prepare_device_tables(p) != SP_OK) return 0;
  return device_layout(*p).total;
}

int sp_plan_bwd_blocks(sp_plan *p, const int32_t **rows, int32_t *n_rows, const int32_t **key_end) {
  if (!p || !rows || !n_rows || !key_end) return SP_ERR_INVALID_ARG;
  if (int rc = prepare_device_tables(p)) return rc;
  *rows = p->bwd_merged.data();
  *n_rows = p->n_bwdm();
  *key_end = p->key_end.data();
  return SP_OK;
}

int sp_plan_upload_to(sp_plan *p, void *device_buffer, size_t buffer_bytes, void *stream) {
  if (!p || !device_buffer) return SP_ERR_INVALID_ARG;
  if (p->d_tiles) return SP_OK;
  if (reinterpret_cast<uintptr_t>(device_buffer) & 255u) return SP_ERR_ALIGNMENT;
  if (int rc = prepare_device_tables(p)) return rc;
  const DeviceLayout l = device_layout(*p);
  if (buffer_bytes < l.total) return SP_ERR_WORKSPACE;
  if (int rc = copy_tables(p, static_cast<char *>(device_buffer), l, static_cast<cudaStream_t>(stream))) {
    p->d_tiles = p->d_ranges = p->d_bwd = p->d_pairs = p->d_pblk = p->d_quads = p->d_qblk = p->d_bwdm =
        p->d_key_end = nullptr;
    return rc;
  }
  p->owns_device = false;
  return SP_OK;
}

void sp_plan_destroy(sp_plan *p) {
  if (!p) return;
  if (p->d_tiles && p->owns_device) cudaFree(p->d_tiles);
  delete p;
}

int sp_tree_attn_fwd(const sp_plan *p, int32_t dtype, const void *q, const void *k, const void *v, void *o,
                     float *lse, int32_t T, int32_t Hq, int32_t Hkv, int32_t D, float softmax_scale,
                     int32_t *d_status, void *stream) {
  if (!p) return SP_ERR_INVALID_ARG;
  if (int rc = check_heads(dtype, T, Hq, Hkv, D)) return rc;
  if (T != p->total_tokens) return SP_ERR_INVALID_ARG;
  if (T == 0) return SP_OK;
  if (!q || !k || !v || !o || !lse) return SP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return SP_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f)) return SP_ERR_INVALID_ARG;
  if (!p->d_tiles) return SP_ERR_NOT_UPLOADED;
  if (!on_plan_device(*p)) return SP_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (int rc = check_tiling(*p, dtype, G)) return rc;
  const spc::AttnShape s{T, Hq, Hkv, D, G, softmax_scale};
  if (dtype == SP_BF16) return spc::tc_fwd(plan_dev(*p), s, q, k, v, o, lse, d_status, stream);
  return spc::simt_fwd(plan_dev(*p), s, dtype, q, k, v, o, lse, d_status, stream);
}

int sp_tree_attn_fwd_paired(const sp_plan *p, int32_t dtype, const void *q, const void *k, const void *v, void *o,
                            float *lse, int32_t T, int32_t Hq, int32_t Hkv, int32_t D, float softmax_scale,
                            int32_t *d_status, void *stream) {
  if (!p) return SP_ERR_INVALID_ARG;
  if (int rc = check_heads(dtype, T, Hq, Hkv, D)) return rc;
  if (dtype != SP_BF16 || D != 128) return SP_ERR_UNSUPPORTED;
  if (T != p->total_tokens) return SP_ERR_INVALID_ARG;
  if (T == 0) return SP_OK;
  if (!q || !k || !v || !o || !lse) return SP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return SP_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f)) return SP_ERR_INVALID_ARG;
  if (!p->d_tiles) return SP_ERR_NOT_UPLOADED;
  if (!on_plan_device(*p)) return SP_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (int rc = check_tiling(*p, dtype, G)) return rc;
  const spc::AttnShape s{T, Hq, Hkv, D, G, softmax_scale};
  return spc::tc_fwd_pair(plan_dev(*p), s, q, k, v, o, lse, d_status, stream);
}

// Workspace: Delta [Hq][T] fp32, then (bf16 only) the fp32 dQ accumulator
// [T][Hq][D] that the tensor-core backward reduces into.
size_t sp_tree_attn_bwd_workspace_bytes(int32_t dtype, int32_t T, int32_t Hq, int32_t D) {
  if (T <= 0 || Hq <= 0 || D <= 0) return 0;
  const size_t delta = align_up(size_t(T) * size_t(Hq) * sizeof(float));
  if (dtype != SP_BF16) return delta;
  return delta + align_up(size_t(T) * size_t(Hq) * size_t(D) * sizeof(float));
}

}  // extern "C"

namespace {

int attn_bwd(const sp_plan *p, int32_t dtype, const void *q, const void *k, const void *v, const void *o,
             const float *lse, const void *d_o, void *dq, void *dk, void *dv, void *workspace, size_t workspace_bytes,
             int32_t T, int32_t Hq, int32_t Hkv, int32_t D, float softmax_scale, bool deterministic,
             int32_t *d_status, void *stream, void *ev_begin = nullptr, void *ev_end = nullptr) {
  if (!p) return SP_ERR_INVALID_ARG;
  if (int rc = check_heads(dtype, T, Hq, Hkv, D)) return rc;
  if (T != p->total_tokens) return SP_ERR_INVALID_ARG;
  if (T == 0) return SP_OK;
  if (!q || !k || !v || !o || !lse || !d_o || !dq || !dk || !dv) return SP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(d_o) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return SP_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f)) return SP_ERR_INVALID_ARG;
  const size_t need = sp_tree_attn_bwd_workspace_bytes(dtype, T, Hq, D);
  if (!workspace || workspace_bytes < need) return SP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return SP_ERR_ALIGNMENT;
  if (!p->d_tiles) return SP_ERR_NOT_UPLOADED;
  if (!on_plan_device(*p)) return SP_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (int rc = check_tiling(*p, dtype, G)) return rc;
  const spc::AttnShape s{T, Hq, Hkv, D, G, softmax_scale};
  float *delta = static_cast<float *>(workspace);
  if (dtype == SP_BF16) {
    float *dqacc = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                             align_up(size_t(T) * size_t(Hq) * sizeof(float)));
    return spc::tc_bwd(plan_dev(*p), s, q, k, v, o, lse, d_o, dq, dk, dv, delta, dqacc, deterministic, d_status,
                       stream, ev_begin, ev_end);
  }
  if (ev_begin || ev_end) return SP_ERR_UNSUPPORTED;  // the fp32 path has no single main kernel
  // the fp32 path computes dQ per query tile already (no atomics)
  return spc::simt_bwd(plan_dev(*p), s, dtype, q, k, v, o, lse, d_o, dq, dk, dv, delta, d_status, stream);
}

}  // namespace

extern "C" {

int sp_tree_attn_bwd(const sp_plan *p, int32_t dtype, const void *q, const void *k, const void *v, const void *o,
                     const float *lse, const void *d_o, void *dq, void *dk, void *dv, void *workspace,
                     size_t workspace_bytes, int32_t T, int32_t Hq, int32_t Hkv, int32_t D, float softmax_scale,
                     int32_t *d_status, void *stream) {
  return attn_bwd(p, dtype, q, k, v, o, lse, d_o, dq, dk, dv, workspace, workspace_bytes, T, Hq, Hkv, D,
                  softmax_scale, false, d_status, stream);
}

int sp_tree_attn_bwd_deterministic(const sp_plan *p, int32_t dtype, const void *q, const void *k, const void *v,
                                   const void *o, const float *lse, const void *d_o, void *dq, void *dk, void *dv,
                                   void *workspace, size_t workspace_bytes, int32_t T, int32_t Hq, int32_t Hkv,
                                   int32_t D, float softmax_scale, int32_t *d_status, void *stream) {
  return attn_bwd(p, dtype, q, k, v, o, lse, d_o, dq, dk, dv, workspace, workspace_bytes, T, Hq, Hkv, D,
                  softmax_scale, true, d_status, stream);
}

int sp_tree_attn_bwd_timed(const sp_plan *p, int32_t dtype, const void *q, const void *k, const void *v,
                           const void *o, const float *lse, const void *d_o, void *dq, void *dk, void *dv,
                           void *workspace, size_t workspace_bytes, int32_t T, int32_t Hq, int32_t Hkv, int32_t D,
                           float softmax_scale, int32_t deterministic, void *ev_main_begin, void *ev_main_end,
                           int32_t *d_status, void *stream) {
  if (deterministic != 0 && deterministic != 1) return SP_ERR_INVALID_ARG;
  return attn_bwd(p, dtype, q, k, v, o, lse, d_o, dq, dk, dv, workspace, workspace_bytes, T, Hq, Hkv, D,
                  softmax_scale, deterministic != 0, d_status, stream, ev_main_begin, ev_main_end);
}

int sp_edge_gather(int32_t dtype, const void *hidden, int32_t T, int32_t hidden_dim, const int32_t *idx, int32_t E,
                   void *out, int32_t *d_status, void *stream) {
  if (dtype != SP_BF16 && dtype != SP_F32) return SP_ERR_UNSUPPORTED;
  if (T < 0 || E < 0 || hidden_dim <= 0) return SP_ERR_INVALID_ARG;
  if (E == 0) return SP_OK;
  if (!hidden || !idx || !out) return SP_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(out)) return SP_ERR_ALIGNMENT;
  return spc::edge_gather(dtype == SP_BF16 ? 2 : 4, hidden, T, hidden_dim, idx, E, out, d_status, stream);
}

size_t sp_edge_gather_bwd_workspace_bytes(int32_t T, int32_t E) {
  if (T < 0 || E < 0) return 0;
  return spc::edge_gather_bwd_workspace(T, E);
}

int sp_edge_gather_bwd(int32_t dtype, const void *grad_out, int32_t E, int32_t hidden_dim, const int32_t *idx,
                       int32_t T, void *grad_hidden, void *workspace, size_t workspace_bytes, int32_t *d_status,
                       void *stream) {
  if (dtype != SP_BF16 && dtype != SP_F32) return SP_ERR_UNSUPPORTED;
  if (T < 0 || E < 0 || hidden_dim <= 0) return SP_ERR_INVALID_ARG;
  if (T == 0) return SP_OK;
  if (!grad_hidden || (E > 0 && (!grad_out || !idx))) return SP_ERR_INVALID_ARG;
  if (hidden_dim % 8) return SP_ERR_UNSUPPORTED;
  if (!aligned16(grad_hidden) || (E > 0 && !aligned16(grad_out))) return SP_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < spc::edge_gather_bwd_workspace(T, E)) return SP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return SP_ERR_ALIGNMENT;
  return spc::edge_gather_bwd(dtype == SP_BF16 ? 2 : 4, grad_out, E, hidden_dim, idx, T, grad_hidden, workspace,
                              d_status, stream);
}

size_t sp_edge_logprob_workspace_bytes(int32_t E, int32_t V) {
  if (E < 0 || V < 1) return 0;
  return spc::lmh_workspace(E, V);
}

int sp_edge_logprob(int32_t dtype, const void *hidden_sel, int32_t E, int32_t Hd, const void *weight, int32_t V,
                    const int32_t *labels, float *logprob, float *lse, void *workspace, size_t workspace_bytes,
                    int32_t *d_status, void *stream) {
  if (dtype != SP_BF16 && dtype != SP_F32) return SP_ERR_INVALID_ARG;
  if (dtype != SP_BF16) return SP_ERR_UNSUPPORTED;
  if (E < 0 || V < 1 || Hd < 1) return SP_ERR_INVALID_ARG;
  if (Hd % 8) return SP_ERR_UNSUPPORTED;
  if (E == 0) return SP_OK;
  if (!hidden_sel || !weight || !labels || !logprob || !lse) return SP_ERR_INVALID_ARG;
  if (!aligned16(hidden_sel) || !aligned16(weight)) return SP_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < spc::lmh_workspace(E, V)) return SP_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return SP_ERR_ALIGNMENT;
  return spc::lmh_fwd(hidden_sel, E, Hd, weight, V, labels, logprob, lse, workspace, d_status, stream);
}

size_t sp_edge_logprob_bwd_workspace_bytes(int32_t E, int32_t V) {
  if (E < 0 || V < 1) return 0;
  return spc::lmh_bwd_workspace(E, V);
}

int sp_edge_logprob_bwd(int32_t dtype, const void *hidden_sel, int32_t E, int32_t Hd, const void *weight, int32_t V,
                        const int32_t *labels, const float *lse, const float *grad_logprob, float *d_hidden_sel,
                        float *d_weight, void *workspace, size_t workspace_bytes, int32_t *d_status, void *stream) {
  if (dtype != SP_BF16 && dtype != SP_F32) return SP_ERR_INVALID_ARG;
  if (dtype != SP_BF16) return SP_ERR_UNSUPPORTED;
  if (E < 0 || V < 1 || Hd < 1) return SP_ERR_INVALID_ARG;
  if (Hd % 8 || V % 8) return SP_ERR_UNSUPPORTED;
  if (!d_hidden_sel && !d_weight) return SP_OK;
  if (!weight || (E > 0 && (!hidden_sel || !labels || !lse || !grad_logprob))) return SP_ERR_INVALID_ARG;
  if (!aligned16(weight) || (E > 0 && !aligned16(hidden_sel)) || (d_hidden_sel && !aligned16(d_hidden_sel)) ||
      (d_weight && !aligned16(d_weight)))
    return SP_ERR_ALIGNMENT;
  if (E == 0) {
    // no actions: the weight gradient is zero
    if (d_weight && cudaMemsetAsync(d_weight, 0, size_t(V) * Hd * sizeof(float),
                                    static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return SP_ERR_CUDA;
    return SP_OK;
  }
  if (!workspace || workspace_bytes < spc::lmh_bwd_workspace(E, V)) return SP_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return SP_ERR_ALIGNMENT;
  return spc::lmh_bwd(hidden_sel, E, Hd, weight, V, labels, lse, grad_logprob, d_hidden_sel, d_weight, workspace,
                      d_status, stream);
}

const char *sp_status_string(int status) {
  switch (status) {
    case SP_OK: return "ok";
    case SP_ERR_INVALID_TREE: return "invalid tree: metadata malformed or not in DFS preorder";
    case SP_ERR_INVALID_ARG: return "invalid argument";
    case SP_ERR_UNSUPPORTED: return "unsupported dtype, head_dim, GQA ratio or plan tiling";
    case SP_ERR_ALIGNMENT: return "tensor pointer not 16-byte aligned";
    case SP_ERR_CUDA: return "CUDA call failed";
    case SP_ERR_TIMEOUT: return "device wait timed out";
    case SP_ERR_INDEX_RANGE: return "edge index out of range";
    case SP_ERR_WORKSPACE: return "workspace missing or too small";
    case SP_ERR_NOT_UPLOADED: return "plan not uploaded to the device";
    case SP_ERR_CAP: return "a root path is longer than the fragment token cap";
    default: return "unknown status";
  }
}

}  // extern "C"
