// dK and dV of tree attention on the sm_103a tensor cores, 128 query rows per
// step (the key-block half of the deterministic backward).
//
// The backward sums every branch's contribution into the prefix the branches
// share (#7914, "feat(hybrid): add opt-in shared-prefix attention and Mamba
// execution", introduction).  In preorder a key is seen exactly by the query
// run [its own position, end of its segment's subtree), so each CTA owns one
// block of 128 keys of one KV head, keeps dK and dV in TMEM and walks that run
// from its end back to the diagonal, 128 query rows at a time (128 / G tokens
// x the G query heads of the KV head).  Per step, recomputing from the saved
// LSE (FlashAttention-style):
//   S^T  = K Q^T,  dP^T = V dO^T                       (SS, N = 128)
//   P^T  = exp(S^T - LSE),  dS^T = P^T (dP^T - Delta)   (8 warps)
//   dV  += P^T dO,  dK += dS^T Q                        (A from TMEM, N = D)
// dQ is not formed here (the per-query-tile kernel forms it without atomics).
//
// Why 128 rows: a tcgen05 product of M = 128 and K = 16 costs about the same
// time at N = 64 as at N = 128 on this part, so 64-row steps run the score
// products at half rate.  128-row steps need S^T and dP^T at 128 columns each;
// with dK and dV that fills the 512 TMEM columns, so P^T and dS^T (bf16 pairs)
// are written over the columns of S^T and dP^T that produced them, and the
// products are ordered so nothing is overwritten early: the tensor pipe runs
// one thread's products in issue order, and the issue order per step is
//   dV(j)  S^T(j+1)  dK(j)  dP^T(j+1)
// (S^T(j+1) after dV(j) has read P^T(j); dP^T(j+1) after dK(j) has read
// dS^T(j)).  The elementwise work of step j+1 splits in two phases that each
// overlap a pair of products: P^T(j+1) as soon as S^T(j+1) is done (while
// dK(j) and dP^T(j+1) run), dS^T(j+1) as soon as dP^T(j+1) is done (while
// dV(j+1) and S^T(j+2) run).  P^T is handed over in two halves of the query
// rows, so dV(j+1) starts on the first half while the second is formed.
//
// Roles: warps 0-7 elementwise, warpgroup h taking query columns [64h, 64h+64)
// of every key row (thread = key row = TMEM lane; its P^T and dS^T go to the
// first 32 of its own 64 columns, so the two warpgroups never write columns
// the other still has to read); warp 8: TMA producer (Q and dO tiles, and each
// step's per-column -LSE and -Delta staged by the whole warp); warp 9: the
// single-thread MMA issuer.  Epilogue: warpgroup 0 stores dK, 1 stores dV.
// Q and dO travel in rings of their own (three and two stages): Q(j) is read
// by S^T(j), the first product of a step, and last by dK(j); dO(j) by dP^T(j)
// and dV(j).  The third Q stage lets Q(j+1) be fetched a whole step before
// S^T(j+1) needs it, which two stages shared by both tiles could not.
// Every mbarrier wait is bounded (Ctl); on expiry the CTA records
// SP_DEV_TIMEOUT, stops issuing, drains, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "pipeline.cuh"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace spc {
namespace {

using namespace ptx;

constexpr int kBK = 128;            // keys per CTA
constexpr int kBQ = 128;            // query rows per step
constexpr int kThreads = 320;       // 8 elementwise warps, producer, MMA
constexpr int kChunk = 128 * 128;   // 128 rows x 128 bytes
constexpr int kQStages = 3;         // Q ring depth
constexpr int kOStages = 2;         // dO ring depth
constexpr int kStatSlots = 2;       // per-step -LSE / -Delta slots
constexpr float kLog2e = 1.4426950408889634f;

enum : int {
  B_KV_FULL = 0,
  B_Q_FULL = 1,     // +stage (3)
  B_Q_EMPTY = 4,    // +stage
  B_O_FULL = 7,     // +stage (2)
  B_O_EMPTY = 9,    // +stage
  B_ST_FULL = 11,   // +slot (2)
  B_ST_EMPTY = 13,  // +slot, 8 warp arrivals
  B_S_FULL = 15,
  B_DP_FULL = 16,
  B_P_FULL = 17,    // +half (2), 8 warp arrivals each
  B_DS_FULL = 19,   // 8 warp arrivals
  B_FINAL = 20,
  B_COUNT = 21
};

// Shared memory: a small region (barriers, TMEM address, abort flag, the
// per-step statistics) first, then the 1024-byte aligned tiles.  At D = 128
// the tiles take 224 KB, so the whole fits the 227 KB a CTA may have only
// when the small region and its padding stay within 3 KB: the kernel checks
// that against the address it was given and reports SP_DEV_SMEM_LAYOUT instead
// of running if not.
template <int D>
struct Layout {
  static constexpr int kDChunks = D / 64;
  static constexpr int TILE = kDChunks * kChunk;  // 128 rows x D
  static constexpr int BAR = 0;
  static constexpr int TSLOT = BAR + 8 * B_COUNT;
  static constexpr int ABORT = TSLOT + 4;
  static constexpr int STAT = (ABORT + 4 + 15) & ~15;  // slot x (-lse2[128], -delta[128])
  static constexpr int MISC = STAT + kStatSlots * 2 * 128 * 4;
  // tile offsets from the aligned tile base
  static constexpr int K = 0;
  static constexpr int V = TILE;
  static constexpr int Q = 2 * TILE;               // + stage * TILE
  static constexpr int DO = Q + kQStages * TILE;   // + stage * TILE
  static constexpr int TILES = DO + kOStages * TILE;
  static constexpr int WANT = ((MISC + 1023) & ~1023) + TILES;
  static constexpr int ALLOC = WANT > 120 * 1024 ? WANT : 120 * 1024;
  static_assert(ALLOC <= 227 * 1024, "shared memory");
};

// TMEM columns: S^T [0, 128) (then P^T), dP^T [128, 256) (then dS^T), dK, dV.
constexpr uint32_t T_S = 0, T_DP = 128, T_DK = 256;

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, PlanDev plan,
                  AttnShape s, const float *__restrict__ lse, const float *__restrict__ delta,
                  __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv, int32_t *d_status, int head_chunk,
                  CtaClock clk) {
  using L = Layout<D>;
  const unsigned long long clk0 = clk.begin();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw;
  const uint32_t sbase = smem_u32(smem);
  // tiles at the first 1024-byte boundary after the small region
  const uint32_t tbase = (sbase + L::MISC + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // key blocks in launch order, head_chunk KV heads at a time (as the
  // 64-row kernel): CTA b runs block (b mod span) / head_chunk of head chunk
  // b / span
  const int span = head_chunk * plan.n_bwdm;
  const int item = (blockIdx.x % span) / head_chunk;
  const int g = (blockIdx.x / span) * head_chunk + blockIdx.x % head_chunk;
  const int *blk = plan.bwdm + 5 * size_t(item);
  const int k0 = blk[1], k1 = blk[2], qb = blk[3], qe = blk[4];
  const int T = s.T;
  if (!(0 <= k0 && k0 < k1 && k1 - k0 <= kBK && qb == k0 && k1 <= qe && qe <= T)) {
    if (threadIdx.x == 0 && d_status) atomicOr(d_status, SP_DEV_BAD_PLAN);
    return;
  }
  if (tbase - sbase + L::TILES > uint32_t(L::ALLOC)) {
    if (threadIdx.x == 0 && d_status) atomicOr(d_status, SP_DEV_SMEM_LAYOUT);
    return;
  }
  constexpr int tps = kBQ / G;  // query tokens per step
  const int nq = (qe - qb + tps - 1) / tps;
  auto q_of = [&](int jj) { return qb + (nq - 1 - jj) * tps; };  // walked from the run's end

  Ctl ctl{sbase + L::BAR, reinterpret_cast<volatile int *>(smem + L::ABORT), d_status, kSpinLimit};
  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(ctl.bar(i), (i == B_P_FULL || i == B_P_FULL + 1 || i == B_DS_FULL || i == B_ST_EMPTY ||
                             i == B_ST_EMPTY + 1) ? 8u : 1u);
    *ctl.abort = 0;
    fence_mbar_init();
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
      mbar_arrive_expect_tx(ctl.bar(B_KV_FULL), 2u * L::TILE);
#pragma unroll
      for (int c = 0; c < L::kDChunks; ++c) {
        tma_load_3d(tbase + L::K + c * kChunk, &tm_k, ctl.bar(B_KV_FULL), c * 64, g, k0);
        tma_load_3d(tbase + L::V + c * kChunk, &tm_v, ctl.bar(B_KV_FULL), c * 64, g, k0);
      }
    }
    // -LSE (log2) and -Delta of a step's 128 columns, loaded one step ahead
    float nl[4], nd[4];
    auto load_stats = [&](int jj) {
      const int qt = q_of(jj);
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int c = lane + 32 * x;
        const int tok = qt + c / G, head = g * G + c % G;
        const bool ok = jj < nq && tok < qe;
        nl[x] = ok ? __ldg(lse + size_t(head) * T + tok) * kLog2e : 0.f;
        nd[x] = ok ? __ldg(delta + size_t(head) * T + tok) : 0.f;
      }
    };
    load_stats(0);
    int nqi = 0, noi = 0;  // Q and dO tiles issued
    for (int j = 0; j < nq; ++j) {
      const int qs = j % kQStages, os = j % kOStages, ss = j % kStatSlots;
      const int qt = q_of(j);
      // Q(j) once S^T(j - 3) and dK(j - 3) have read its stage
      if (!ctl.wait_warp(B_Q_EMPTY + qs, ((j / kQStages) & 1) ^ 1)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(ctl.bar(B_Q_FULL + qs), L::TILE);
#pragma unroll
        for (int c = 0; c < L::kDChunks; ++c)
          tma_load_3d(tbase + L::Q + qs * L::TILE + c * kChunk, &tm_q, ctl.bar(B_Q_FULL + qs), c * 64, g * G, qt);
      }
      ++nqi;
      // dO(j) once dP^T(j - 2) and dV(j - 2) have read its stage
      if (!ctl.wait_warp(B_O_EMPTY + os, ((j / kOStages) & 1) ^ 1)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(ctl.bar(B_O_FULL + os), L::TILE);
#pragma unroll
        for (int c = 0; c < L::kDChunks; ++c)
          tma_load_3d(tbase + L::DO + os * L::TILE + c * kChunk, &tm_do, ctl.bar(B_O_FULL + os), c * 64, g * G, qt);
      }
      ++noi;
      // the step's statistics once the elementwise warps are done with step j - 2
      if (!ctl.wait_warp(B_ST_EMPTY + ss, ((j / kStatSlots) & 1) ^ 1)) break;
      float *stat = reinterpret_cast<float *>(smem + L::STAT + ss * 2 * 128 * 4);
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        stat[lane + 32 * x] = -nl[x];
        stat[kBQ + lane + 32 * x] = -nd[x];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(ctl.bar(B_ST_FULL + ss));
      load_stats(j + 1);
    }
    if (lane == 0 && *ctl.abort) {
      ctl.drain(B_KV_FULL, 0);
      for (int m = nqi - kQStages < 0 ? 0 : nqi - kQStages; m < nqi; ++m)
        ctl.drain(B_Q_FULL + m % kQStages, (m / kQStages) & 1);
      for (int m = noi - kOStages < 0 ? 0 : noi - kOStages; m < noi; ++m)
        ctl.drain(B_O_FULL + m % kOStages, (m / kOStages) & 1);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(kBK, kBQ, 0, 0);  // S^T, dP^T
      constexpr uint32_t id_kv = idesc_bf16_f32(kBK, D, 0, 1);   // dV, dK (B MN-major)
      const uint64_t dk_kmaj = smem_desc_sw128(tbase + L::K, 16, 1024);
      const uint64_t dv_kmaj = smem_desc_sw128(tbase + L::V, 16, 1024);
      auto q_tile = [&](int jj) { return tbase + L::Q + (jj % kQStages) * L::TILE; };
      auto o_tile = [&](int jj) { return tbase + L::DO + (jj % kOStages) * L::TILE; };
      // S^T(j) = K Q^T or dP^T(j) = V dO^T, K = D
      auto issue_scores = [&](uint32_t dcol, uint64_t a, uint32_t b_addr) {
        const uint64_t b = smem_desc_sw128(b_addr, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + dcol, a + off, b + off, id_s, kk > 0);
        }
      };
      // dV or dK += (P^T or dS^T from TMEM) (dO or Q, MN-major), K = 128 query rows.
      // Warpgroup h left its 64 columns' bf16 pairs in the first 32 of its 64
      // TMEM columns, so query rows [64h, 64h + 64) sit at column 64h + (row - 64h) / 2.
      auto issue_grad = [&](uint32_t dcol, uint32_t acol, uint32_t b_addr, bool acc) {
        const uint64_t b = smem_desc_sw128(b_addr, kChunk, 1024);
#pragma unroll
        for (int kk = 0; kk < kBQ / 16; ++kk)
          mma_bf16_ts(tmem + dcol, tmem + acol + 64 * (kk >> 2) + 8 * (kk & 3), b + ((kk * 2048) >> 4), id_kv,
                      (acc || kk > 0));
      };
      // the same product over the K steps of one half of each group's columns:
      // half x covers query rows 64h + 32x + [0, 32), K steps 4h + 2x and 4h + 2x + 1
      auto issue_grad_half = [&](uint32_t dcol, uint32_t acol, uint32_t b_addr, int x, bool acc) {
        const uint64_t b = smem_desc_sw128(b_addr, kChunk, 1024);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int kk = 4 * (i >> 1) + 2 * x + (i & 1);
          mma_bf16_ts(tmem + dcol, tmem + acol + 64 * (kk >> 2) + 8 * (kk & 3), b + ((kk * 2048) >> 4), id_kv,
                      (acc || i > 0));
        }
      };
      bool ok = ctl.wait(B_KV_FULL, 0) && ctl.wait(B_Q_FULL, 0);
      if (ok) {
        tc_fence_after();
        issue_scores(T_S, dk_kmaj, q_tile(0));
        mma_commit(ctl.bar(B_S_FULL));
      }
      if (ok && (ok = ctl.wait(B_O_FULL, 0))) {
        tc_fence_after();
        issue_scores(T_DP, dv_kmaj, o_tile(0));
        mma_commit(ctl.bar(B_DP_FULL));
      }
      for (int j = 0; ok && j < nq; ++j) {
        // dV += P^T dO, each half of the query rows as soon as its P^T is in TMEM
        if (!(ok = ctl.wait(B_P_FULL, j & 1))) break;
        tc_fence_after();
        issue_grad_half(T_DK + D, T_S, o_tile(j), 0, j > 0);
        if (!(ok = ctl.wait(B_P_FULL + 1, j & 1))) break;
        tc_fence_after();
        issue_grad_half(T_DK + D, T_S, o_tile(j), 1, true);
        mma_commit(ctl.bar(B_O_EMPTY + j % kOStages));  // dO(j): dP^T(j) and dV(j) done
        if (j + 1 < nq) {
          if (!(ok = ctl.wait(B_Q_FULL + (j + 1) % kQStages, ((j + 1) / kQStages) & 1))) break;
          tc_fence_after();
          issue_scores(T_S, dk_kmaj, q_tile(j + 1));  // after dV(j) read P^T(j)
          mma_commit(ctl.bar(B_S_FULL));
        }
        if (!(ok = ctl.wait(B_DS_FULL, j & 1))) break;
        tc_fence_after();
        issue_grad(T_DK, T_DP, q_tile(j), j > 0);  // dK += dS^T Q
        mma_commit(ctl.bar(B_Q_EMPTY + j % kQStages));
        if (j + 1 < nq) {
          if (!(ok = ctl.wait(B_O_FULL + (j + 1) % kOStages, ((j + 1) / kOStages) & 1))) break;
          tc_fence_after();
          issue_scores(T_DP, dv_kmaj, o_tile(j + 1));  // after dK(j) read dS^T(j)
          mma_commit(ctl.bar(B_DP_FULL));
        }
      }
      mma_commit(ctl.bar(B_FINAL));
      ctl.drain(B_FINAL, 0);
    }
  } else {
    // ---------------------------------------------------- P^T and dS^T (8 warps)
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
    for (int j = 0; j < nq; ++j) {
      const int ss = j % kStatSlots;
      const int qt = q_of(j);
      const float *stat = reinterpret_cast<const float *>(smem + L::STAT + ss * 2 * 128 * 4);
      const bool nomask = qt + tps <= key_qe && qt >= k1 - 1;
      const int kq = key - qt;  // column c is visible iff kq <= c / G and its token < key_qe
      const int ql = key_qe - qt;  // tokens of this step inside this key's query run
      if (!(ok = ctl.wait_warp(B_ST_FULL + ss, (j / kStatSlots) & 1))) break;  // the step's statistics
      if (!(ok = ctl.wait_warp(B_S_FULL, j & 1))) break;
      tc_fence_after();
      // phase A: P^T of this group's 64 columns in two halves of 32, each
      // released as soon as it is in TMEM (dV starts on the first); P is kept
      // in fp32 for phase B
      float pv[64];
      uint32_t us[64];
      tmem_ld32x2(tmem + lane_base + T_S + 64 * h, tmem + lane_base + T_S + 64 * h + 32,
                  *reinterpret_cast<uint32_t(*)[32]>(us), *reinterpret_cast<uint32_t(*)[32]>(us + 32));
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float4 *nl4 = reinterpret_cast<const float4 *>(stat) + 16 * h + 8 * half;
        float nl2[32];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 a = nl4[q4];
          nl2[4 * q4] = a.x, nl2[4 * q4 + 1] = a.y, nl2[4 * q4 + 2] = a.z, nl2[4 * q4 + 3] = a.w;
        }
        float *p = pv + 32 * half;
        const uint32_t *u = us + 32 * half;
        if (nomask && kvalid) {
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            ffma2(p[i], p[i + 1], __uint_as_float(u[i]), __uint_as_float(u[i + 1]), sl2, sl2, nl2[i], nl2[i + 1]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int c = 64 * h + 32 * half + i;
            const bool vis = kvalid && c / G < ql && kq <= c / G;
            p[i] = vis ? fmaf(__uint_as_float(u[i]), sl2, nl2[i]) : -INFINITY;
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) p[i] = ex2(p[i]);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(p[2 * i], p[2 * i + 1]);
        // over the first 32 of this group's S^T columns (all of them read above)
        tmem_st16(tmem + lane_base + T_S + 64 * h + 16 * half, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ctl.bar(B_P_FULL + half));
      }
      // phase B: dS^T = P^T (dP^T - Delta)
      if (!(ok = ctl.wait_warp(B_DP_FULL, j & 1))) break;
      tc_fence_after();
      uint32_t dsk[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t ud[32];
        tmem_ld32(tmem + lane_base + T_DP + 64 * h + 32 * half, ud);
        const float4 *nd4 = reinterpret_cast<const float4 *>(stat + kBQ) + 16 * h + 8 * half;
        float ndl[32];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 a = nd4[q4];
          ndl[4 * q4] = a.x, ndl[4 * q4 + 1] = a.y, ndl[4 * q4 + 2] = a.z, ndl[4 * q4 + 3] = a.w;
        }
        const float *p = pv + 32 * half;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float t0, t1, d0, d1;
          fadd2(t0, t1, __uint_as_float(ud[i]), __uint_as_float(ud[i + 1]), ndl[i], ndl[i + 1]);
          fmul2(d0, d1, p[i], p[i + 1], t0, t1);
          dsk[16 * half + i / 2] = pack_bf16(d0, d1);
        }
      }
      tmem_st32(tmem + lane_base + T_DP + 64 * h, dsk);  // over the first 32 of this group's dP^T columns
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(ctl.bar(B_DS_FULL));
        mbar_arrive(ctl.bar(B_ST_EMPTY + ss));  // this step's statistics are read
      }
    }
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

template <int D, int G>
int launch(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, const float *lse,
           const void *d_o, void *dk, void *dv, const float *delta, int head_chunk, int32_t *d_status,
           cudaStream_t st, cudaEvent_t ev_begin, cudaEvent_t ev_end) {
  CUtensorMap tq, tdo, tk, tv;
  int rc = encode_bf16_3d(&tq, q, D, s.Hq, s.T, 64, G, kBQ / G);
  if (!rc) rc = encode_bf16_3d(&tdo, d_o, D, s.Hq, s.T, 64, G, kBQ / G);
  if (!rc) rc = encode_bf16_3d(&tk, k, D, s.Hkv, s.T, 64, 1, kBK);
  if (!rc) rc = encode_bf16_3d(&tv, v, D, s.Hkv, s.T, 64, 1, kBK);
  if (rc) return rc;
  auto kern = bwd_kv_kernel<D, G>;
  const int smem = Layout<D>::ALLOC;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return SP_ERR_CUDA;
  CtaClock clk;
  cta_clock_for(kClockKeyBlocks, &clk.buf, &clk.cap);
  const unsigned grid = unsigned(p.n_bwdm) * unsigned(s.Hkv);
  if (ev_begin && cudaEventRecord(ev_begin, st) != cudaSuccess) return SP_ERR_CUDA;
  kern<<<grid, kThreads, smem, st>>>(tq, tdo, tk, tv, p, s, lse, delta, static_cast<__nv_bfloat16 *>(dk),
                                     static_cast<__nv_bfloat16 *>(dv), d_status, head_chunk, clk);
  if (cudaGetLastError() != cudaSuccess) return SP_ERR_CUDA;
  if (ev_end && cudaEventRecord(ev_end, st) != cudaSuccess) return SP_ERR_CUDA;
  return SP_OK;
}

}  // namespace

int tc_bwd_kv(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, const float *lse,
              const void *d_o, void *dk, void *dv, const float *delta, int head_chunk, int32_t *d_status,
              void *stream, void *ev_begin, void *ev_end) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaEvent_t e0 = static_cast<cudaEvent_t>(ev_begin), e1 = static_cast<cudaEvent_t>(ev_end);
#define SPC_KV_CASE(DD, GG)                                                                               \
  if (s.D == DD && s.G == GG)                                                                             \
    return launch<DD, GG>(p, s, q, k, v, lse, d_o, dk, dv, delta, head_chunk, d_status, st, e0, e1);
  SPC_KV_CASE(64, 1) SPC_KV_CASE(64, 2) SPC_KV_CASE(64, 4) SPC_KV_CASE(64, 8)
  SPC_KV_CASE(128, 1) SPC_KV_CASE(128, 2) SPC_KV_CASE(128, 4) SPC_KV_CASE(128, 8)
#undef SPC_KV_CASE
  return SP_ERR_UNSUPPORTED;
}

}  // namespace spc
