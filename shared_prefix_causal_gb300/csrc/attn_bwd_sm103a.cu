// Tree attention backward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// The backward sums every branch's contribution into the prefix the branches
// share (#7914, "feat(hybrid): add opt-in shared-prefix attention and Mamba
// execution", introduction).  In preorder, the queries that can see a key are
// exactly the key's own later tokens and every token of its segment's
// subtree: one contiguous run [kv_start, subtree end).  So each CTA owns one
// block of 128 keys of one KV head, keeps dK and dV for it in TMEM, and walks
// that query run in 64-row blocks (64 / G tokens x the G query heads of the
// KV head).  Every child branch below a prefix adds into the same TMEM
// accumulators; nothing is scattered.  Per query block, FlashAttention-style
// recomputation from the saved LSE:
//   S^T  = K Q^T          dP^T = V dO^T                    (tensor cores)
//   P^T  = exp(S^T - LSE) dS^T = P^T (dP^T - Delta)        (8 warps)
//   dV  += P^T dO         dK  += dS^T Q                    (tensor cores)
//   dQ^T = K^T dS^T  -> fp32 atomics into the dQ workspace (4 of the 8 warps)
// dQ is formed transposed (M = head_dim) so it needs only 64 TMEM columns:
// S^T, dP^T, dQ^T, two P^T buffers, dK and dV fill the 512 columns.
//
// Roles: warps 0-7 form P^T and dS^T, warpgroup h taking query columns
// [32h, 32h + 32) of every key row (TMEM lane = key row); warps 4-7 also read
// dQ^T out (TMEM lane = head-dim index); in the epilogue warps 0-3 store dK
// and warps 4-7 dV.  Warp 8: TMA producer (Q, dO, and the per-column LSE /
// Delta staged by the whole warp); warps 9 and 10: one MMA issuer each, warp 9
// for S^T and dP^T, warp 10 for dV, dK and dQ^T.  S^T and dP^T of block j are
// issued as soon as block j-1's have been read, so the elementwise work of
// block j overlaps the gradient products of block j-1.  The two issuers share
// the tensor pipe but wait on their own barriers: an mbarrier wait costs the
// waiting thread about a hundred cycles even when the phase is complete, and a
// thread blocked there issues nothing, so one issuer's waits run while the
// other's products keep the pipe busy.  Their products write disjoint TMEM
// columns and every operand they share is handed over through barriers (P^T,
// dS^T and dQ^T double- or single-buffered with full/free pairs, a Q/dO stage
// released by warp 10 after the products that read it last), so no ordering
// between the two threads' products is needed.
//
// Companion kernels (attn_bwd_pre_sm103a.cu): bwd_pre (Delta = rowsum(dO * O)
// and zeroing the fp32 dQ workspace) and dq_convert (scale and round dQ to
// bf16).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "pipeline.cuh"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace spc {
namespace {

using namespace ptx;

constexpr int kBK = 128;            // keys per CTA
constexpr int kBQ = 64;             // query rows per block
constexpr int kThreads = 352;       // 11 warps
constexpr int kKChunk = 128 * 128;  // 128 rows x 128 bytes
constexpr int kQChunk = 64 * 128;   // 64 rows x 128 bytes
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kStages = 3;  // Q/dO ring depth

enum : int {
  B_KV_FULL = 0,
  B_Q_FULL = 1,    // +stage (3)
  B_Q_EMPTY = 4,   // +stage
  B_S_FULL = 7,
  B_S_FREE = 8,
  B_P_FULL = 9,    // +buffer (2)
  B_P_FREE = 11,   // +buffer
  B_DQ_FULL = 13,
  B_DQ_FREE = 14,
  B_FINAL = 15,
  B_SDP_DONE = 16,  // the S^T / dP^T issuer's last products have completed
  B_COUNT = 17
};

template <int D>
struct Layout {
  static constexpr int kDChunks = D / 64;
  // K keeps two 64-column chunks even for D = 64 (the second one zeroed) so
  // that dQ^T = K^T dS^T always runs as an M = 128 MMA.
  static constexpr int K = 0;
  static constexpr int V = K + 2 * kKChunk;
  static constexpr int STAGE = V + kDChunks * kKChunk;
  static constexpr int Q_OFF = 0;                          // within a stage
  static constexpr int DO_OFF = kDChunks * kQChunk;
  static constexpr int STAT_OFF = 2 * kDChunks * kQChunk;  // lse2[64], delta[64]
  static constexpr int STAGE_BYTES = STAT_OFF + 1024;     // keep 1024-byte alignment
  static constexpr int PS = STAGE + kStages * STAGE_BYTES;  // two dS^T buffers
  static constexpr int PS_BYTES = kKChunk;
  static constexpr int BAR = PS + 2 * PS_BYTES;
  static constexpr int TSLOT = BAR + 8 * B_COUNT;
  static constexpr int ABORT = TSLOT + 4;
  static constexpr int BYTES = ABORT + 4 + 1024;
  static constexpr int ALLOC = BYTES > 120 * 1024 ? BYTES : 120 * 1024;
  static constexpr uint32_t QTILE_BYTES = kDChunks * kQChunk;  // one of Q / dO for a block
};

// TMEM columns: S^T, dP^T (fp32, 64 each), dQ^T (fp32, 64), two P^T buffers
// (bf16 pairs, 32 each), dK and dV (fp32, D each; 256 + 2D <= 512)
constexpr uint32_t T_S = 0, T_DP = 64, T_DQ = 128, T_P = 192, T_DK = 256;


template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, PlanDev plan,
                  AttnShape s, const float *__restrict__ lse, const float *__restrict__ delta,
                  float *__restrict__ dqacc, __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv,
                  int32_t *d_status, int head_chunk, CtaClock clk) {
  using L = Layout<D>;
  const unsigned long long clk0 = clk.begin();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived by pointer arithmetic so that accesses
  // through it stay shared-memory (not generic) accesses
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Key blocks in launch order (grouped by query-run end), head_chunk KV heads
  // at a time: CTA b runs block (b mod head_chunk*n_bwd) / head_chunk of head
  // chunk b / (head_chunk*n_bwd).
  const int span = head_chunk * plan.n_bwdm;
  const int item = (blockIdx.x % span) / head_chunk;
  const int g = (blockIdx.x / span) * head_chunk + blockIdx.x % head_chunk;
  const int *blk = plan.bwdm + 5 * item;
  const int k0 = blk[1], k1 = blk[2], qb = blk[3], qe = blk[4];
  const int T = s.T, Hq = s.Hq;
  if (!(0 <= k0 && k0 < k1 && k1 - k0 <= kBK && qb == k0 && k1 <= qe && qe <= T)) {
    if (threadIdx.x == 0 && d_status) atomicOr(d_status, SP_DEV_BAD_PLAN);
    return;
  }
  constexpr int tpb = kBQ / G;  // query tokens per block
  const int nq = (qe - qb + tpb - 1) / tpb;
  // The run is walked from its end back to the diagonal block: CTAs whose runs
  // end at the same subtree end then read the same Q/dO rows and add into the
  // same dQ rows at about the same time, while those rows are in L2.
  auto q_of = [&](int jj) { return qb + (nq - 1 - jj) * tpb; };

  Ctl ctl{sbase + L::BAR, reinterpret_cast<volatile int *>(smem + L::ABORT), d_status, kSpinLimit};
  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      if (i == B_S_FREE || i == B_P_FULL || i == B_P_FULL + 1) cnt = 256;  // warps 0-7, every thread
      if (i == B_DQ_FREE) cnt = 256;                                       // warps 0-7
      mbar_init(ctl.bar(i), cnt);
    }
    *ctl.abort = 0;
    fence_mbar_init();
  }
  if (D == 64 && warp < 4) {
    // zero the padding chunk of K (read by the M = 128 dQ^T MMA)
    uint4 *z = reinterpret_cast<uint4 *>(smem + L::K + kKChunk);
    for (int i = threadIdx.x; i < kKChunk / 16; i += 128) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 9) {
    tmem_alloc(sbase + L::TSLOT, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::TSLOT);

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_do);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(ctl.bar(B_KV_FULL), 2u * L::kDChunks * kKChunk);
#pragma unroll
      for (int c = 0; c < L::kDChunks; ++c) {
        tma_load_3d(sbase + L::K + c * kKChunk, &tm_k, ctl.bar(B_KV_FULL), c * 64, g, k0);
        tma_load_3d(sbase + L::V + c * kKChunk, &tm_v, ctl.bar(B_KV_FULL), c * 64, g, k0);
      }
    }
    // LSE (as log2) and Delta of the next block's 64 columns, loaded one block
    // ahead so their latency hides behind the ring wait.
    float nl[2], nd[2];
    auto load_stats = [&](int jj) {
      const int qt = q_of(jj);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = lane + 32 * h;
        const int tok = qt + c / G, head = g * G + c % G;
        const bool ok = jj < nq && tok < qe;
        nl[h] = ok ? __ldg(lse + size_t(head) * T + tok) * kLog2e : 0.f;
        nd[h] = ok ? __ldg(delta + size_t(head) * T + tok) : 0.f;
      }
    };
    load_stats(0);
    int j = 0;
    for (; j < nq; ++j) {
      const int st = j % kStages;
      if (!ctl.wait_warp(B_Q_EMPTY + st, ((j / kStages) & 1) ^ 1)) break;
      const int qt = q_of(j);
      const uint32_t stage = L::STAGE + st * L::STAGE_BYTES;
      if (lane == 0) {
        // byte count first, copies next, the one arrival after the stats below
        mbar_expect_tx(ctl.bar(B_Q_FULL + st), 2u * L::QTILE_BYTES);
#pragma unroll
        for (int c = 0; c < L::kDChunks; ++c) {
          tma_load_3d(sbase + stage + L::Q_OFF + c * kQChunk, &tm_q, ctl.bar(B_Q_FULL + st), c * 64, g * G, qt);
          tma_load_3d(sbase + stage + L::DO_OFF + c * kQChunk, &tm_do, ctl.bar(B_Q_FULL + st), c * 64, g * G, qt);
        }
      }
      float *stat = reinterpret_cast<float *>(smem + stage + L::STAT_OFF);
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // staged negated: the consumers add them
        stat[lane + 32 * h] = -nl[h];
        stat[kBQ + lane + 32 * h] = -nd[h];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(ctl.bar(B_Q_FULL + st));
      load_stats(j + 1);
    }
    if (lane == 0 && *ctl.abort) {
      ctl.drain(B_KV_FULL, 0);
      for (int m = j - kStages < 0 ? 0 : j - kStages; m < j; ++m)
        ctl.drain(B_Q_FULL + m % kStages, (m / kStages) & 1);
    }
  } else if (warp == 9) {
    // ----------------------------------------------- S^T and dP^T MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(kBK, kBQ, 0, 0);  // S^T, dP^T
      // operand descriptors, built once; a K step only moves the start address
      const uint64_t dk_kmaj = smem_desc_sw128(sbase + L::K, 16, 1024);
      const uint64_t dv_kmaj = smem_desc_sw128(sbase + L::V, 16, 1024);
      bool ok = ctl.wait(B_KV_FULL, 0);
      tc_fence_after();
      for (int j = 0; ok && j < nq; ++j) {
        const int st = j % kStages;
        const uint32_t stage = sbase + L::STAGE + st * L::STAGE_BYTES;
        if (!(ok = ctl.wait(B_Q_FULL + st, (j / kStages) & 1))) break;
        if (!(ok = ctl.wait(B_S_FREE, (j & 1) ^ 1))) break;
        tc_fence_after();
        const uint64_t dq_k = smem_desc_sw128(stage + L::Q_OFF, 16, 1024);
        const uint64_t ddo_k = smem_desc_sw128(stage + L::DO_OFF, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ka = ((kk >> 2) * kKChunk + (kk & 3) * 32) >> 4;
          const uint32_t qa = ((kk >> 2) * kQChunk + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + T_S, dk_kmaj + ka, dq_k + qa, id_s, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ka = ((kk >> 2) * kKChunk + (kk & 3) * 32) >> 4;
          const uint32_t qa = ((kk >> 2) * kQChunk + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + T_DP, dv_kmaj + ka, ddo_k + qa, id_s, kk > 0);
        }
        mma_commit(ctl.bar(B_S_FULL));
      }
      // every product of this thread has completed before TMEM is freed
      mma_commit(ctl.bar(B_SDP_DONE));
      ctl.drain(B_SDP_DONE, 0);
    }
  } else if (warp == 10) {
    // ------------------------------------------ dV, dK and dQ^T MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_kv = idesc_bf16_f32(kBK, D, 0, 1);   // dV, dK
      constexpr uint32_t id_q = idesc_bf16_f32(128, kBQ, 1, 1);  // dQ^T
      const uint64_t dk_mn = smem_desc_sw128(sbase + L::K, kKChunk, 1024);
      // per dS^T buffer b: dS^T as A (K-major) and as B (MN-major)
      const uint64_t dst_kmaj0 = smem_desc_sw128(sbase + L::PS, 16, 1024);
      const uint64_t dst_mn0 = smem_desc_sw128(sbase + L::PS, kQChunk, 1024);
      constexpr uint32_t kPsStep = uint32_t(L::PS_BYTES) >> 4;  // descriptor units between buffers
      // P^T(m) in TMEM implies S^T(m), and so K, V and the stage's Q/dO, were
      // in shared memory; K/V and the stage are still checked
      bool ok = ctl.wait(B_KV_FULL, 0);
      for (int m = 0; ok && m < nq; ++m) {
        const int st = m % kStages, pb = m & 1;
        const uint32_t stage = sbase + L::STAGE + st * L::STAGE_BYTES;
        if (!(ok = ctl.wait(B_P_FULL + pb, (m >> 1) & 1))) break;
        if (!(ok = ctl.wait(B_Q_FULL + st, (m / kStages) & 1))) break;
        tc_fence_after();
        const uint64_t ddo_mn = smem_desc_sw128(stage + L::DO_OFF, kQChunk, 1024);
        const uint32_t pso = pb * kPsStep;
        const uint64_t dst_kmaj = dst_kmaj0 + pso, dst_mn = dst_mn0 + pso;
        const uint64_t dq_mn = smem_desc_sw128(stage + L::Q_OFF, kQChunk, 1024);
        // dV += P^T dO (P^T read from TMEM, 8 columns per K step); dK += dS^T Q  (K = 64 query rows)
#pragma unroll
        for (int kk = 0; kk < kBQ / 16; ++kk)
          mma_bf16_ts(tmem + T_DK + D, tmem + T_P + 32 * pb + 8 * kk, ddo_mn + ((kk * 2048) >> 4), id_kv,
                      (m > 0 || kk > 0));
#pragma unroll
        for (int kk = 0; kk < kBQ / 16; ++kk)
          mma_bf16_ss(tmem + T_DK, dst_kmaj + ((kk * 32) >> 4), dq_mn + ((kk * 2048) >> 4), id_kv, (m > 0 || kk > 0));
        // dV and dK were the stage's last readers (S^T(m) and dP^T(m) completed
        // before P^T(m) existed): release it before waiting for the dQ^T buffer
        mma_commit(ctl.bar(B_Q_EMPTY + st));
        if (!(ok = ctl.wait(B_DQ_FREE, (m & 1) ^ 1))) break;
        tc_fence_after();
        // dQ^T = K^T dS^T   (K = 128 keys)
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          mma_bf16_ss(tmem + T_DQ, dk_mn + ((kk * 2048) >> 4), dst_mn + ((kk * 2048) >> 4), id_q, kk > 0);
        mma_commit(ctl.bar(B_DQ_FULL));
        mma_commit(ctl.bar(B_P_FREE + pb));
      }
      mma_commit(ctl.bar(B_FINAL));
      ctl.drain(B_FINAL, 0);
    }
  } else {
    // ------------------------------ P^T, dS^T (+ dQ readout, dK/dV epilogue)
    // Two warpgroups split each 64-query block by columns: group h (warps
    // 4h..4h+3) handles query columns [32h, 32h + 32) of every key row (thread
    // = key row = TMEM lane).  Both load their S^T and dP^T columns at once, so
    // S_FREE (and the next block's S^T/dP^T products) follows right away.
    // After handing over block j's P^T and dS^T each group reads its half of
    // block j-1's dQ^T out of TMEM and adds it into the fp32 workspace; in the
    // epilogue group 0 stores dK and group 1 dV.
    const int h = warp >> 2;
    const int r = threadIdx.x & 127;  // key row = TMEM lane
    const uint32_t lane_base = uint32_t(32 * (warp & 3)) << 16;
    const int key = k0 + r;
    const bool kvalid = key < k1;
    // this key's own run end: a block may hold keys of segments of its first
    // key's subtree, seen by fewer of the run's queries
    const int key_qe = kvalid ? min(plan.key_end[key], qe) : qb;
    const float sl2 = s.scale * kLog2e;
    bool ok = true;
    // dQ^T of block m: TMEM lane d = head-dim index, 64 query columns; one
    // fp32 atomic add per (column, d) into the workspace row of that query
    // Block m's dQ^T out of TMEM and into the fp32 workspace: warpgroup h
    // takes query columns [32h, 32h + 32) (tokens 32h / G on), so the
    // reductions are shared by all eight warps.
    auto dq_readout = [&](int m) -> bool {
      const int qt = q_of(m) + 32 * h / G;
      if (!ctl.wait_warp(B_DQ_FULL, m & 1)) return false;
      tc_fence_after();
      uint32_t u[32];
      tmem_ld32(tmem + lane_base + T_DQ + 32 * h, u);
      tc_fence_before();
      mbar_arrive(ctl.bar(B_DQ_FREE));
      const int d = r;
      if (d < D) {
        // query column 32h + c is token qt + c / G, head g * G + c % G
        float *base = dqacc + (size_t(qt) * Hq + g * G) * D + d;
        const size_t tstride = size_t(Hq) * D;
        if (q_of(m) + tpb <= qe) {
#pragma unroll
          for (int c = 0; c < 32; ++c) atomicAdd(base + (c / G) * tstride + (c % G) * D, __uint_as_float(u[c]));
        } else {
          const int ql = qe - qt;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c / G < ql) atomicAdd(base + (c / G) * tstride + (c % G) * D, __uint_as_float(u[c]));
        }
      }
      return true;
    };
    for (int j = 0; ok && j < nq; ++j) {
      const int st = j % kStages;
      const int qt = q_of(j);
      const float *stat = reinterpret_cast<const float *>(smem + L::STAGE + st * L::STAGE_BYTES + L::STAT_OFF);
      if (!(ok = ctl.wait_warp(B_Q_FULL + st, (j / kStages) & 1))) break;
      if (!(ok = ctl.wait_warp(B_S_FULL, j & 1))) break;
      tc_fence_after();
      const int pb = j & 1;
      const uint32_t prow = sbase + L::PS + pb * L::PS_BYTES + r * 128;
      const bool nomask = qt + tpb <= key_qe && qt >= k1 - 1;
      const int kq = key - qt;  // column c is visible iff kq <= c / G and its token < key_qe
      const int ql = key_qe - qt;  // tokens of this block inside this key's query run
      uint32_t us[32], ud[32];
      tmem_ld32x2(tmem + lane_base + T_S + 32 * h, tmem + lane_base + T_DP + 32 * h, us, ud);
      tc_fence_before();
      mbar_arrive(ctl.bar(B_S_FREE));
      // this group's -LSE (log2) and -Delta, as float4 shared loads
      float nl2[32], ndl[32];
      const float4 *st4 = reinterpret_cast<const float4 *>(stat);
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 a = st4[8 * h + q4], b = st4[16 + 8 * h + q4];
        nl2[4 * q4] = a.x, nl2[4 * q4 + 1] = a.y, nl2[4 * q4 + 2] = a.z, nl2[4 * q4 + 3] = a.w;
        ndl[4 * q4] = b.x, ndl[4 * q4 + 1] = b.y, ndl[4 * q4 + 2] = b.z, ndl[4 * q4 + 3] = b.w;
      }
      // phases: exponents (masked to -inf), all exp2 back to back, products;
      // paired fp32 instructions where the columns need no test
      float pv[32], dsv[32];
      if (nomask && kvalid) {  // two loops: a per-column test inside one loop is far slower
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          ffma2(pv[i], pv[i + 1], __uint_as_float(us[i]), __uint_as_float(us[i + 1]), sl2, sl2, nl2[i],
                nl2[i + 1]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = 32 * h + i;
          const bool vis = kvalid && c / G < ql && kq <= c / G;
          pv[i] = vis ? fmaf(__uint_as_float(us[i]), sl2, nl2[i]) : -INFINITY;
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) pv[i] = ex2(pv[i]);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float t0, t1;
        fadd2(t0, t1, __uint_as_float(ud[i]), __uint_as_float(ud[i + 1]), ndl[i], ndl[i + 1]);
        fmul2(dsv[i], dsv[i + 1], pv[i], pv[i + 1], t0, t1);
      }
      if (!(ok = ctl.wait_warp(B_P_FREE + pb, ((j >> 1) & 1) ^ 1))) break;  // block j-2's MMAs done
      {  // P^T: this group's 32 query columns as 16 bf16 pairs into this row's TMEM lane
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(pv[2 * i], pv[2 * i + 1]);
        tmem_st16(tmem + lane_base + T_P + 32 * pb + 16 * h, pk);
      }
#pragma unroll
      for (int u4 = 0; u4 < 4; ++u4) {  // dS^T: K-major, 128-byte swizzle
        const int u8 = 4 * h + u4;
        const float *y = dsv + 8 * u4;
        const uint32_t off = (u8 ^ (r & 7)) << 4;
        st_shared_v4(prow + off, pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                     pack_bf16(y[6], y[7]));
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ctl.bar(B_P_FULL + pb));
      if (j >= 1 && !(ok = dq_readout(j - 1))) break;
    }
    if (ok && nq >= 1) ok = dq_readout(nq - 1);
    if (ok && ctl.wait_warp(B_FINAL, 0)) {
      tc_fence_after();
      // group 0: dK (scaled); group 1: dV
      __nv_bfloat16 *dst = (h == 0 ? dk : dv) + (size_t(key) * s.Hkv + g) * D;
      const float mul = h == 0 ? s.scale : 1.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_base + T_DK + h * D + 32 * c, u);
        if (kvalid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(u[i]) * mul, __uint_as_float(u[i + 1]) * mul);
            w.y = pack_bf16(__uint_as_float(u[i + 2]) * mul, __uint_as_float(u[i + 3]) * mul);
            w.z = pack_bf16(__uint_as_float(u[i + 4]) * mul, __uint_as_float(u[i + 5]) * mul);
            w.w = pack_bf16(__uint_as_float(u[i + 6]) * mul, __uint_as_float(u[i + 7]) * mul);
            *reinterpret_cast<uint4 *>(dst + 32 * c + i) = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  clk.end(clk0);
}

// How many KV heads' key blocks run together.  Fewer heads in flight means
// fewer distinct Q/dO/dQ rows, so CTAs walking the same query run share them
// through L2; but a chunk must hold enough work that its longest query run does
// not finish long after the rest.  Pick the smallest divisor c of Hkv for which
// a chunk's average work per SM is at least twice the longest run, in query
// blocks plus a fixed per-CTA cost.
int bwd_head_chunk(const PlanDev &p, const AttnShape &s, int sms) {
  const double tpb = double(kBQ / s.G), fixed = 6.0;
  const double total = double(p.bwdm_run_sum) / tpb + fixed * p.n_bwdm;
  const double longest = double(p.bwdm_run_max) / tpb + fixed;
  for (int c = 1; c < s.Hkv; ++c)
    if (s.Hkv % c == 0 && c * total / double(sms) >= 2.0 * longest) return c;
  return s.Hkv;
}

template <int D, int G>
int launch(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, const void *o,
           const float *lse, const void *d_o, void *dq, void *dk, void *dv, float *delta, float *dqacc,
           bool deterministic, int32_t *d_status, cudaStream_t st, cudaEvent_t ev_begin, cudaEvent_t ev_end) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long rows = long(s.T) * s.Hq;
  if (int rc0 = bwd_pre(s, o, d_o, delta, deterministic ? nullptr : dqacc, sms, st)) return rc0;

  CUtensorMap tq, tdo, tk, tv;
  int rc = encode_bf16_3d(&tq, q, D, s.Hq, s.T, 64, G, kBQ / G);
  if (!rc) rc = encode_bf16_3d(&tdo, d_o, D, s.Hq, s.T, 64, G, kBQ / G);
  if (!rc) rc = encode_bf16_3d(&tk, k, D, s.Hkv, s.T, 64, 1, kBK);
  if (!rc) rc = encode_bf16_3d(&tv, v, D, s.Hkv, s.T, 64, 1, kBK);
  if (rc) return rc;
  const int head_chunk = bwd_head_chunk(p, s, sms);
  if (deterministic) {
    // dK, dV by the 128-row key-block kernel; dQ without atomics: every query
    // tile walks its own key blocks
    const int rc2 = tc_bwd_kv(p, s, q, k, v, lse, d_o, dk, dv, delta, head_chunk, d_status, st, ev_begin, ev_end);
    if (rc2) return rc2;
    return tc_dq(p, s, q, k, v, lse, d_o, dq, delta, d_status, st);
  }
  auto kern = bwd_tc_kernel<D, G>;
  const int smem = Layout<D>::ALLOC;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return SP_ERR_CUDA;
  const unsigned grid = unsigned(p.n_bwdm) * unsigned(s.Hkv);
  if (ev_begin && cudaEventRecord(ev_begin, st) != cudaSuccess) return SP_ERR_CUDA;
  CtaClock clk;
  cta_clock_for(kClockKeyBlocks, &clk.buf, &clk.cap);
  kern<<<grid, kThreads, smem, st>>>(tq, tdo, tk, tv, p, s, lse, delta, dqacc, static_cast<__nv_bfloat16 *>(dk),
                                     static_cast<__nv_bfloat16 *>(dv), d_status, head_chunk, clk);
  if (cudaGetLastError() != cudaSuccess) return SP_ERR_CUDA;
  if (ev_end && cudaEventRecord(ev_end, st) != cudaSuccess) return SP_ERR_CUDA;

  return dq_convert(dqacc, dq, s.scale, rows * D, sms, st);
}

}  // namespace

int tc_bwd(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, const void *o,
           const float *lse, const void *d_o, void *dq, void *dk, void *dv, float *delta, float *dqacc,
           bool deterministic, int32_t *d_status, void *stream, void *ev_begin, void *ev_end) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaEvent_t e0 = static_cast<cudaEvent_t>(ev_begin), e1 = static_cast<cudaEvent_t>(ev_end);
#define SPC_BWD_CASE(DD, GG)                                                                          \
  if (s.D == DD && s.G == GG)                                                                         \
    return launch<DD, GG>(p, s, q, k, v, o, lse, d_o, dq, dk, dv, delta, dqacc, deterministic, d_status, st, e0, e1);
  SPC_BWD_CASE(64, 1) SPC_BWD_CASE(64, 2) SPC_BWD_CASE(64, 4) SPC_BWD_CASE(64, 8)
  SPC_BWD_CASE(128, 1) SPC_BWD_CASE(128, 2) SPC_BWD_CASE(128, 4) SPC_BWD_CASE(128, 8)
#undef SPC_BWD_CASE
  return SP_ERR_UNSUPPORTED;
}

}  // namespace spc
