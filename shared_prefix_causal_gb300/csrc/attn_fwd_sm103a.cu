// Tree attention forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes: for every query token, softmax attention over the keys of
// its ancestor segments (all visible) and of its own segment up to itself
// (causal): each query segment attends causally over its ancestors (PR #7387
// "TreePackedSeqParams", "Summary"; issue #7386, "Describe the solution
// you'd like": each query run attends only to its ancestor path).
// Outputs O (bf16) and the natural-log LSE (fp32) kept for the backward.
//
// One CTA per (pair of query tiles, KV head).  A tile is 128 rows = (128 / G)
// tokens x the G query heads sharing that KV head, so every K/V block read
// from L2 or HBM feeds full 128-row MMAs even for short segments.  The two
// tiles of a pair are neighbours in the plan's schedule (tile k of sibling
// segments, or consecutive tiles of one segment): they share their ancestor
// blocks, so the CTA streams the merged list of 128-key blocks once.
//   warp 8  (one lane)  TMA producer: both Q tiles once, then K and V blocks
//                       into a two-stage ring;
//   warp 9  (one lane)  MMA issuer, interleaving the tiles so one tile's
//                       softmax overlaps the other tile's MMAs:
//                         PV_a(n), S_a(n+1), PV_b(n), S_b(n+1), ...
//                       S = Q K^T goes to the tile's TMEM S columns; the
//                       softmax overwrites them with P (bf16 pairs) and
//                       O += P V reads P straight from TMEM;
//   warps 0-3 / 4-7     softmax of tile a / tile b: thread r owns row r (TMEM
//                       lane r).  Masks only where needed (range tail; causal
//                       only on blocks that reach past the tile's first
//                       token), exp2-domain online softmax with a lazily
//                       updated reference max (O is rescaled in TMEM only when
//                       the row max grows by more than 2^8), epilogue O / l.
// TMEM: S_a, O_a, S_b, O_b (128 columns each for D = 128).  tcgen05 MMAs of
// one thread execute in issue order, so S(n+1) never overwrites P(n) before
// PV(n) has read it, and the commit that signals S(n+1) also covers PV(n):
// the softmax always sees a complete O when it rescales.
// Every mbarrier wait is bounded; on expiry the CTA records SP_DEV_TIMEOUT,
// stops issuing work, drains what it issued, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "pipeline.cuh"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace spc {
namespace {

using namespace ptx;

constexpr int kBM = 128;           // query rows per tile
constexpr int kBN = 128;           // keys per block
constexpr int kStages = 2;         // K/V ring depth
constexpr int kThreads = 384;      // 8 softmax warps + producer + MMA + 2 idle (a full third warpgroup)
// Registers: the launch gives every thread 168; the third warpgroup (producer,
// MMA, idle) drops to kRegsIssue and the softmax warpgroups take what it
// frees: 2 x 128 x kRegsSoftmax + 128 x kRegsIssue = 384 x 168.
constexpr int kRegsIssue = 136;
constexpr int kRegsSoftmax = 184;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsIssue <= kThreads * 168, "register split");
constexpr int kChunk = 128 * 128;  // bytes of one 128-row x 128-byte swizzled chunk
constexpr int kRunsInSmem = 128;  // block runs of a work item kept in shared memory
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum : int {
  B_Q_FULL = 0,
  B_K_FULL = 1,    // +stage
  B_K_EMPTY = 3,   // +stage
  B_V_FULL = 5,    // +stage
  B_V_EMPTY = 7,   // +stage
  B_S_FULL = 9,    // +tile
  B_P_FULL = 11,   // +tile (128 arrivals)
  B_O_DONE = 13,   // +tile (one completion per P V of that tile)
  B_MMA_DONE = 15,
  B_COUNT = 16
};

template <int D>
struct Layout {
  static constexpr int kDChunks = D / 64;
  static constexpr int KV = kDChunks * kChunk;  // bytes of 128 rows x D
  static constexpr int Q = 0;                   // + tile * KV
  static constexpr int K = 2 * KV;              // + stage * KV
  static constexpr int V = K + kStages * KV;
  static constexpr int RUNS = V + kStages * KV;  // the work item's block runs (kRunsInSmem x 32 bytes)
  static constexpr int BAR = RUNS + kRunsInSmem * 32;
  static constexpr int TSLOT = BAR + 8 * B_COUNT;
  static constexpr int ABORT = TSLOT + 4;
  static constexpr int BYTES = ABORT + 4 + 1024;  // + alignment slack
  // at least ~116 KB so two CTAs never share an SM (each takes all 512 TMEM columns)
  static constexpr int ALLOC = BYTES > 120 * 1024 ? BYTES : 120 * 1024;
  static constexpr uint32_t TILE_COLS = 128 + D;  // S then O, per tile
};


template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, PlanDev plan, AttnShape s,
                  __nv_bfloat16 *__restrict__ o, float *__restrict__ lse, int32_t *d_status, CtaClock clk) {
  using L = Layout<D>;
  const unsigned long long clk0 = clk.begin();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived by pointer arithmetic so that accesses
  // through it stay shared-memory (not generic) accesses
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int g = blockIdx.x / plan.n_pairs;
  const int *pr = plan.pairs + 4 * size_t(blockIdx.x % plan.n_pairs);
  const int ta = pr[0], tb = pr[1], rbeg = pr[2], nrun = pr[3];
  const int G = s.G, T = s.T;
  const int *runs = plan.pblk + 8 * size_t(rbeg);  // the pair's runs of key blocks (slot 0: a, 1: b)

  // Validate the work item (uniform over the CTA).
  bool bad = !(0 <= ta && ta < plan.n_tiles && -1 <= tb && tb < plan.n_tiles && nrun >= 1);
  const int *tla = plan.tiles + 5 * size_t(bad ? 0 : ta);
  const int *tlb = !bad && tb >= 0 ? plan.tiles + 5 * size_t(tb) : nullptr;
  const int qa0 = tla[1], qa1 = tla[2];
  const int qb0 = tlb ? tlb[1] : 0, qb1 = tlb ? tlb[2] : 0;
  bad = bad || !(0 <= qa0 && qa0 < qa1 && qa1 <= T && (!tlb || (0 <= qb0 && qb0 < qb1 && qb1 <= T)));
  const int64_t blocks = bad ? -1 : check_runs(runs, nrun, T, tlb ? 3u : 1u);
  const int nblk = int(blocks);
  if (blocks < 1 || blocks > (int64_t(1) << 30)) bad = true;
  if (bad) {
    if (threadIdx.x == 0 && d_status) atomicOr(d_status, SP_DEV_BAD_PLAN);
    return;
  }

  Ctl ctl{sbase + L::BAR, reinterpret_cast<volatile int *>(smem + L::ABORT), d_status, kSpinLimit};
  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(ctl.bar(i), (i == B_P_FULL || i == B_P_FULL + 1) ? 128u : 1u);
    *ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(sbase + L::TSLOT, 512);
    tmem_relinquish();
  }
  // The work item's runs are read by every role at every block: from shared
  // memory when they fit (they do unless a tile's ranges split into many runs)
  const bool runs_in_smem = nrun <= kRunsInSmem;
  if (runs_in_smem) {
    int32_t *dst = reinterpret_cast<int32_t *>(smem + L::RUNS);
    for (int i = threadIdx.x; i < 8 * nrun; i += kThreads) dst[i] = runs[i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::TSLOT);
  if (runs_in_smem) runs = reinterpret_cast<const int32_t *>(smem + L::RUNS);
  if (warp >= 8) {
    // third warpgroup: producer, MMA issuer, two idle warps
    setmaxnreg_dec<kRegsIssue>();
    if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(ctl.bar(B_Q_FULL), (tlb ? 2u : 1u) * L::KV);
#pragma unroll
      for (int c = 0; c < L::kDChunks; ++c) {
        tma_load_3d(sbase + L::Q + c * kChunk, &tm_q, ctl.bar(B_Q_FULL), c * 64, g * G, qa0);
        if (tlb) tma_load_3d(sbase + L::Q + L::KV + c * kChunk, &tm_q, ctl.bar(B_Q_FULL), c * 64, g * G, qb0);
      }
      int n = 0;
      RunCursor cur(runs);
      for (; n < nblk; ++n, cur.next()) {
        const int st = n & 1, kb = cur.kb();
        const uint32_t ph = (n >> 1) & 1;
        if (!ctl.wait(B_K_EMPTY + st, ph ^ 1)) break;
        mbar_arrive_expect_tx(ctl.bar(B_K_FULL + st), L::KV);
#pragma unroll
        for (int c = 0; c < L::kDChunks; ++c)
          tma_load_3d(sbase + L::K + st * L::KV + c * kChunk, &tm_k, ctl.bar(B_K_FULL + st), c * 64, g, kb);
        if (!ctl.wait(B_V_EMPTY + st, ph ^ 1)) {
          ctl.drain(B_K_FULL + st, ph);
          break;
        }
        mbar_arrive_expect_tx(ctl.bar(B_V_FULL + st), L::KV);
#pragma unroll
        for (int c = 0; c < L::kDChunks; ++c)
          tma_load_3d(sbase + L::V + st * L::KV + c * kChunk, &tm_v, ctl.bar(B_V_FULL + st), c * 64, g, kb);
      }
      if (*ctl.abort) {
        // let the last fills of each stage land before the CTA exits
        ctl.drain(B_Q_FULL, 0);
        for (int m = n - 2 < 0 ? 0 : n - 2; m < n; ++m) {
          ctl.drain(B_K_FULL + (m & 1), (m >> 1) & 1);
          ctl.drain(B_V_FULL + (m & 1), (m >> 1) & 1);
        }
      }
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, 0, 1);
      // operand descriptors, built once; a K step only moves the start address
      const uint64_t dq_a = smem_desc_sw128(sbase + L::Q, 16, 1024);
      const uint64_t dq_b = smem_desc_sw128(sbase + L::Q + L::KV, 16, 1024);
      const uint64_t dk_s0 = smem_desc_sw128(sbase + L::K, 16, 1024);
      const uint64_t dk_s1 = smem_desc_sw128(sbase + L::K + L::KV, 16, 1024);
      const uint64_t dv_s0 = smem_desc_sw128(sbase + L::V, kChunk, 1024);
      const uint64_t dv_s1 = smem_desc_sw128(sbase + L::V + L::KV, kChunk, 1024);
      uint32_t pcount_a = 0, pcount_b = 0;  // P V issued per tile
      // S_t(n) = Q_t K_n^T into tile t's S columns
      auto issue_s = [&](int t, int n) {
        const uint64_t dk = (n & 1) ? dk_s1 : dk_s0;
        const uint64_t dq = t ? dq_b : dq_a;
        const uint32_t tsc = tmem + t * L::TILE_COLS;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tsc, dq + off, dk + off, idesc_s, kk > 0);
        }
        mma_commit(ctl.bar(B_S_FULL + t));
      };
      // O_t += P_t(n) V_n with P read from tile t's S columns
      auto issue_pv = [&](int t, int n, bool accumulate) {
        const uint64_t dv = (n & 1) ? dv_s1 : dv_s0;
        const uint32_t tsc = tmem + t * L::TILE_COLS;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_bf16_ts(tsc + 128, tsc + 8 * kk, dv + ((kk * 2048) >> 4), idesc_o, (accumulate || kk > 0));
        mma_commit(ctl.bar(B_O_DONE + t));
      };
      RunCursor cur(runs), nxt(runs);  // blocks n and n + 1
      bool ok = ctl.wait(B_Q_FULL, 0) && ctl.wait(B_K_FULL, 0);
      if (ok) {
        tc_fence_after();
        if (cur.end(0)) issue_s(0, 0);
        if (cur.end(1)) issue_s(1, 0);
        mma_commit(ctl.bar(B_K_EMPTY));
        if (nblk > 1) nxt.next();
      }
      for (int n = 0; ok && n < nblk; ++n) {
        const int st = n & 1;
        const bool last = n + 1 == nblk;
        const bool ua = cur.end(0) != 0, ub = cur.end(1) != 0;
        const bool ua1 = !last && nxt.end(0) != 0, ub1 = !last && nxt.end(1) != 0;
        if (!last) cur.next();
        if (n + 2 < nblk) nxt.next();
        if (!(ok = ctl.wait(B_V_FULL + st, (n >> 1) & 1))) break;
        if (ua) {
          if (!(ok = ctl.wait(B_P_FULL, pcount_a & 1))) break;
          tc_fence_after();
          issue_pv(0, n, pcount_a > 0);
          ++pcount_a;
        }
        // block n+1's K tile: needed from here on
        if (!last && !(ok = ctl.wait(B_K_FULL + (st ^ 1), ((n + 1) >> 1) & 1))) break;
        tc_fence_after();
        if (ua1) issue_s(0, n + 1);
        if (ub) {
          if (!(ok = ctl.wait(B_P_FULL + 1, pcount_b & 1))) break;
          tc_fence_after();
          issue_pv(1, n, pcount_b > 0);
          ++pcount_b;
        }
        if (ub1) issue_s(1, n + 1);
        if (!last) mma_commit(ctl.bar(B_K_EMPTY + (st ^ 1)));
        mma_commit(ctl.bar(B_V_EMPTY + st));
      }
      mma_commit(ctl.bar(B_MMA_DONE));
      ctl.drain(B_MMA_DONE, 0);
    }
    }
  } else {
    // ------------------------------------------------------------- softmax
    setmaxnreg_inc<kRegsSoftmax>();
    const int t = warp >> 2;  // tile handled by this warpgroup
    const int r = threadIdx.x & 127;
    const bool active = t == 0 || tlb != nullptr;
    const uint32_t lane_base = uint32_t(32 * (warp & 3)) << 16;
    const uint32_t ts = tmem + t * L::TILE_COLS + lane_base;  // this row's S (then P) columns; O at +128
    const int q0 = t ? qb0 : qa0, q1 = t ? qb1 : qa1;
    const int rows_valid = (q1 - q0) * G;
    const int tok = q0 + r / G;
    const int head = g * G + r % G;
    const float sl2 = s.scale * kLog2e;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    uint32_t used = 0;  // blocks this tile has processed
    RunCursor cur(runs);
    for (int n = 0; active && n < nblk; ++n, cur.next()) {
      const int kb = cur.kb(), kv1 = cur.end(t);
      if (kv1 == 0) continue;
      const bool causal = cur.causal(t);
      if (!(ok = ctl.wait_warp(B_S_FULL + t, used & 1))) break;
      tc_fence_after();
      float sv[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 64; ++c) {
        uint32_t u0[32], u1[32];
        tmem_ld32x2(ts + 64 * c, ts + 64 * c + 32, u0, u1);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          sv[64 * c + j] = __uint_as_float(u0[j]);
          sv[64 * c + 32 + j] = __uint_as_float(u1[j]);
        }
      }
      // row max of the raw scores (masked ones set to -inf) by a tree of 8
      // partials; the scale is applied to the max (it is positive)
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
      const bool full = kb + kBN <= kv1 && (!causal || kb + kBN - 1 <= q0);
      if (!full) {
        const int lim = causal ? min(kv1 - kb, tok - kb + 1) : kv1 - kb;
#pragma unroll
        for (int j = 0; j < kBN; ++j) sv[j] = j < lim ? sv[j] : -INFINITY;
      }
      // three-input maxima: two new scores per instruction
#pragma unroll
      for (int j = 0; j < kBN; j += 2) mx[(j >> 1) & 7] = fmax3(mx[(j >> 1) & 7], sv[j], sv[j + 1]);
      const float mb = sl2 * fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      const float m_new = (mb > m_run + kRescaleThreshold) ? mb : m_run;
      const float mref = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ex2(m_run - mref);
      // exponents with one FFMA each, then all exponentials back to back, then
      // a tree sum and P as bf16 pairs over the first 64 S columns (read by
      // the P V MMA)
      const float nm = -mref;
      // paired fp32 arithmetic: one instruction per two scores
#pragma unroll
      for (int j = 0; j < kBN; j += 2) ffma2(sv[j], sv[j + 1], sv[j], sv[j + 1], sl2, sl2, nm, nm);
#pragma unroll
      for (int j = 0; j < kBN; ++j) sv[j] = ex2(sv[j]);
      float sm[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) sm[i] = 0.f;
#pragma unroll
      for (int j = 0; j < kBN; j += 2) {
        const int i = (j >> 1) & 3;
        fadd2(sm[2 * i], sm[2 * i + 1], sm[2 * i], sm[2 * i + 1], sv[j], sv[j + 1]);
      }
      l_run = l_run * alpha + (((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7])));
      m_run = m_new;
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(sv[32 * c + 2 * i], sv[32 * c + 2 * i + 1]);
        tmem_st16(ts + 16 * c, pk);
      }
      // O already holds every earlier block (see the header note): rescale it
      // in TMEM, 64 columns at a time, when any row of the warp needs it (P is
      // stored first so its registers are free).
      if (used > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t u0[32], u1[32];
          const uint32_t ta_ = ts + 128 + 64 * c;
          tmem_ld32x2(ta_, ta_ + 32, u0, u1);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            u0[j] = __float_as_uint(__uint_as_float(u0[j]) * alpha);
            u1[j] = __float_as_uint(__uint_as_float(u1[j]) * alpha);
          }
          tmem_st32(ta_, u0);
          tmem_st32(ta_ + 32, u1);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(ctl.bar(B_P_FULL + t));
      ++used;
    }
    if (active && ok && used > 0 && ctl.wait_warp(B_O_DONE + t, (used - 1) & 1)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const bool store = r < rows_valid;
      __nv_bfloat16 *orow = o + (size_t(tok) * s.Hq + head) * D;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t u0[32], u1[32];
        tmem_ld32x2(ts + 128 + 64 * c, ts + 128 + 64 * c + 32, u0, u1);
        if (store) {
#pragma unroll
          for (int j = 0; j < 64; j += 8) {
            const uint32_t *u = j < 32 ? u0 + j : u1 + (j - 32);
            uint4 w;
            w.x = pack_bf16(__uint_as_float(u[0]) * inv, __uint_as_float(u[1]) * inv);
            w.y = pack_bf16(__uint_as_float(u[2]) * inv, __uint_as_float(u[3]) * inv);
            w.z = pack_bf16(__uint_as_float(u[4]) * inv, __uint_as_float(u[5]) * inv);
            w.w = pack_bf16(__uint_as_float(u[6]) * inv, __uint_as_float(u[7]) * inv);
            *reinterpret_cast<uint4 *>(orow + 64 * c + j) = w;
          }
        }
      }
      if (store) lse[size_t(head) * T + tok] = (m_run + log2f(l_run)) * kLn2;
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

template <int D>
int launch(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, void *o, float *lse,
           int32_t *d_status, cudaStream_t st) {
  if (!p.pairs || p.n_pairs <= 0) return SP_ERR_NOT_UPLOADED;
  CUtensorMap tq, tk, tv;
  const int G = s.G;
  int rc = encode_bf16_3d(&tq, q, D, s.Hq, s.T, 64, G, kBM / G);
  if (!rc) rc = encode_bf16_3d(&tk, k, D, s.Hkv, s.T, 64, 1, kBN);
  if (!rc) rc = encode_bf16_3d(&tv, v, D, s.Hkv, s.T, 64, 1, kBN);
  if (rc) return rc;
  auto kern = fwd_tc_kernel<D>;
  const int smem = Layout<D>::ALLOC;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return SP_ERR_CUDA;
  // setmaxnreg.inc waits until the registers it asks for are free: launch only
  // if the block's registers at launch cover the split, or it would never return
  static int regs = 0;
  if (!regs) {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return SP_ERR_CUDA;
    regs = fa.numRegs;
  }
  if (regs * kThreads < 2 * 128 * kRegsSoftmax + 128 * kRegsIssue) return SP_ERR_UNSUPPORTED;
  const unsigned grid = unsigned(p.n_pairs) * unsigned(s.Hkv);
  CtaClock clk;
  cta_clock_for(kClockForward, &clk.buf, &clk.cap);
  kern<<<grid, kThreads, smem, st>>>(tq, tk, tv, p, s, static_cast<__nv_bfloat16 *>(o), lse, d_status, clk);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

}  // namespace

int tc_fwd(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, void *o, float *lse,
           int32_t *d_status, void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return s.D == 64 ? launch<64>(p, s, q, k, v, o, lse, d_status, st)
                   : launch<128>(p, s, q, k, v, o, lse, d_status, st);
}

}  // namespace spc
