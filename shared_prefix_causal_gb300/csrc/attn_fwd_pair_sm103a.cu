// Tree attention forward on a pair of SMs (tcgen05 cta_group::2 + TMEM + TMA).
//
// Computes what fwd_tc_kernel computes -- each query token's softmax attention
// over its ancestor segments' keys (all visible) and its own segment's keys
// up to itself (PR #7387 "TreePackedSeqParams", "Summary"; issue #7386,
// "Describe the solution you'd like": each query run attends only to its
// ancestor path) -- with the two CTAs of a cluster acting as one MMA unit.
//
// Why: with one SM, a 128 x 128 x 16 product reads 8 KB of operands from
// shared memory, as many bytes per cycle as shared memory delivers, so the
// forward's products run below the tensor pipe's rate whenever TMA fills or
// other traffic share the port.  Over a pair, S = Q K^T runs as M = 256 (each
// SM's 128 query rows of A) with each SM holding half of the key block's rows
// of B, and O += P V with P from each SM's TMEM and each SM holding half of
// V's head-dim columns: per SM the products read 6 KB (S) and 2 KB (P V) per
// step, and each SM loads only half of every K and V block.
//
// Work item: a quad of four query tiles (128 rows each: (128 / G) tokens x the
// G query heads of one KV head) and the merged list of their 128-key blocks.
// Slot a holds two consecutive tiles of one segment (offsets 2i, 2i + 1: the
// same key blocks up to one), the even CTA's tile in the M = 256 product's
// first half; slot b the next such couple in the schedule (couple i of a
// sibling segment).  As in the one-SM kernel the two slots ping-pong so one
// slot's softmax overlaps the other slot's products.
//   warp 8, each CTA      TMA producer: its own Q tiles, then its half of every
//                         K block (64 keys) and V block (64 head-dim columns)
//                         into a four-stage ring; completions are counted on
//                         the even CTA's barriers;
//   warp 9, even CTA      MMA issuer for the pair; commits signal both CTAs;
//   warp 9, both          TMEM allocation for the pair;
//   warps 0-3 / 4-7       softmax of the CTA's slot-a / slot-b tile, thread =
//                         row = TMEM lane, exactly as in the one-SM kernel; a
//                         block the slot reads but this CTA's tile does not
//                         gets P = 0 and leaves the row statistics alone.
// TMEM per CTA: S_a, O_a, S_b, O_b (128 columns each).  head_dim 128 only (the
// V half is one 64-column swizzle atom); head_dim 64 uses the one-SM kernel.
// Every mbarrier wait is bounded; on expiry the CTA records SP_DEV_TIMEOUT and
// winds down.  Both CTAs always reach both cluster barriers, so neither can
// leave while the other may still signal its barriers or read its memory.
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

constexpr int D = 128;             // head_dim of this kernel
constexpr int kBN = 128;           // keys per block
constexpr int kStages = 4;         // K/V ring depth
constexpr int kThreads = 320;      // 8 softmax warps + producer + MMA
constexpr int kChunk = 128 * 128;  // one 128-row x 128-byte swizzled chunk (Q)
constexpr int kHalfChunk = 64 * 128;  // 64 rows x 128 bytes (this CTA's K half, per head-dim chunk)
constexpr int kRunsInSmem = 128;  // block runs of a work item kept in shared memory
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum : int {
  B_Q_FULL = 0,    // even CTA: both CTAs' Q tiles
  B_K_FULL = 1,    // +stage (4), even CTA: both halves
  B_K_EMPTY = 5,   // +stage, both CTAs
  B_V_FULL = 9,    // +stage, even CTA: both halves
  B_V_EMPTY = 13,  // +stage, both CTAs
  B_S_FULL = 17,   // +slot, both CTAs
  B_P_FULL = 19,   // +slot, even CTA: 4 warps x 2 CTAs
  B_O_DONE = 21,   // +slot, both CTAs
  B_MMA_DONE = 23,
  B_COUNT = 24
};

struct Layout {
  static constexpr int QT = 2 * kChunk;       // one Q tile: 128 rows x 128 head dims
  static constexpr int KH = 2 * kHalfChunk;   // this CTA's K half: 64 keys x 128 head dims
  static constexpr int VH = kChunk;           // this CTA's V half: 128 keys x 64 head dims
  static constexpr int Q = 0;                 // + slot * QT
  static constexpr int K = 2 * QT;            // + stage * KH
  static constexpr int V = K + kStages * KH;  // + stage * VH
  static constexpr int RUNS = V + kStages * VH;  // the work item's block runs (kRunsInSmem x 32 bytes)
  static constexpr int BAR = RUNS + kRunsInSmem * 32;
  static constexpr int TSLOT = BAR + 8 * B_COUNT;
  static constexpr int ABORT = TSLOT + 4;
  static constexpr int BYTES = ABORT + 4 + 1024;  // + alignment slack
  static constexpr uint32_t TILE_COLS = 128 + D;  // S then O, per slot
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, PlanDev plan, AttnShape s,
                    __nv_bfloat16 *__restrict__ o, float *__restrict__ lse, int32_t *d_status, CtaClock clk) {
  using L = Layout;
  const unsigned long long clk0 = clk.begin();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  const int cl = blockIdx.x >> 1;
  const int g = cl / plan.n_quads;
  const int *qd = plan.quads + 6 * size_t(cl % plan.n_quads);
  const int rbeg = qd[4], nrun = qd[5];
  const int *runs = plan.qblk + 8 * size_t(rbeg);  // the quad's runs of key blocks (slots a0, a1, b0, b1)
  const int G = s.G, T = s.T;
  int t4[4], q0s[4], q1s[4];

  // Validate the work item: both CTAs read the same entries and so take the
  // same decision (neither reaches a cluster barrier the other skips).
  bool bad = nrun < 1 || qd[0] < 0;
  for (int i = 0; i < 4; ++i) {
    t4[i] = qd[i];
    q0s[i] = q1s[i] = 0;
    if (t4[i] >= plan.n_tiles || t4[i] < -1) bad = true;
    if (!bad && t4[i] >= 0) {
      q0s[i] = plan.tiles[5 * size_t(t4[i]) + 1];
      q1s[i] = plan.tiles[5 * size_t(t4[i]) + 2];
      if (!(0 <= q0s[i] && q0s[i] < q1s[i] && q1s[i] <= T)) bad = true;
    }
  }
  uint32_t present = 0;
  for (int i = 0; i < 4; ++i) present |= t4[i] >= 0 ? (1u << i) : 0u;
  const int64_t blocks = bad ? -1 : check_runs(runs, nrun, T, present);
  const int nblk = int(blocks);
  if (blocks < 1 || blocks > (int64_t(1) << 30)) bad = true;
  if (bad) {
    if (threadIdx.x == 0 && leader && d_status) atomicOr(d_status, SP_DEV_BAD_PLAN);
    return;
  }

  Ctl ctl{sbase + L::BAR, reinterpret_cast<volatile int *>(smem + L::ABORT), d_status, kSpinLimit};
  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(ctl.bar(i), (i == B_P_FULL || i == B_P_FULL + 1) ? 8u : 1u);
    *ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc_pair(sbase + L::TSLOT, 512);
    tmem_relinquish_pair();
  }
  // The work item's runs are read by every role at every block: from shared
  // memory when they fit (they do unless a tile's ranges split into many runs)
  const bool runs_in_smem = nrun <= kRunsInSmem;
  if (runs_in_smem) {
    int32_t *dst = reinterpret_cast<int32_t *>(smem + L::RUNS);
    for (int i = threadIdx.x; i < 8 * nrun; i += kThreads) dst[i] = runs[i];
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::TSLOT);
  if (runs_in_smem) runs = reinterpret_cast<const int32_t *>(smem + L::RUNS);
  auto lead_bar = [&](int i) { return mapa_shared(ctl.bar(i), 0); };

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      if (leader) {
        uint32_t tiles = 0;
        for (int i = 0; i < 4; ++i) tiles += t4[i] >= 0 ? 1u : 0u;
        mbar_arrive_expect_tx(ctl.bar(B_Q_FULL), tiles * uint32_t(L::QT));
      }
      for (int slot = 0; slot < 2; ++slot) {
        const int i = 2 * slot + int(rank);
        if (t4[i] < 0) continue;
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_load_3d_pair(sbase + L::Q + slot * L::QT + c * kChunk, &tm_q, lead_bar(B_Q_FULL), c * 64, g * G,
                           q0s[i]);
      }
      int n = 0;
      RunCursor cur(runs);
      for (; n < nblk; ++n, cur.next()) {
        const int st = n % kStages, kb = cur.kb();
        const uint32_t ph = (n / kStages) & 1;
        if (!ctl.wait(B_K_EMPTY + st, ph ^ 1)) break;
        if (leader) mbar_arrive_expect_tx(ctl.bar(B_K_FULL + st), 2u * L::KH);
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_load_3d_pair(sbase + L::K + st * L::KH + c * kHalfChunk, &tm_k, lead_bar(B_K_FULL + st), c * 64, g,
                           kb + 64 * int(rank));
        if (!ctl.wait(B_V_EMPTY + st, ph ^ 1)) break;
        if (leader) mbar_arrive_expect_tx(ctl.bar(B_V_FULL + st), 2u * L::VH);
        tma_load_3d_pair(sbase + L::V + st * L::VH, &tm_v, lead_bar(B_V_FULL + st), 64 * int(rank), g, kb);
      }
      if (*ctl.abort && leader) {
        // let the fills still in flight (this CTA's and the peer's) land
        ctl.drain(B_Q_FULL, 0);
        for (int m = n - kStages < 0 ? 0 : n - kStages; m < n; ++m) {
          ctl.drain(B_K_FULL + m % kStages, (m / kStages) & 1);
          ctl.drain(B_V_FULL + m % kStages, (m / kStages) & 1);
        }
      }
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issuer
    if (leader && lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(256, kBN, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(256, D, 0, 1);
      const uint64_t dq0 = smem_desc_sw128(sbase + L::Q, 16, 1024);
      const uint64_t dq1 = smem_desc_sw128(sbase + L::Q + L::QT, 16, 1024);
      uint32_t pcount[2] = {0, 0};  // P V issued per slot
      // whether a slot reads the block under a cursor
      auto used = [&](int slot, const RunCursor &c) { return (c.end(2 * slot) | c.end(2 * slot + 1)) != 0; };
      // S_slot(n) = Q_slot K_n^T into the slot's S columns of both CTAs
      auto issue_s = [&](int slot, int n) {
        const uint64_t dk = smem_desc_sw128(sbase + L::K + (n % kStages) * L::KH, 16, 1024);
        const uint64_t dq = slot ? dq1 : dq0;
        const uint32_t tsc = tmem + slot * L::TILE_COLS;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qa = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
          const uint32_t ka = ((kk >> 2) * kHalfChunk + (kk & 3) * 32) >> 4;
          mma_pair_ss(tsc, dq + qa, dk + ka, idesc_s, kk > 0);
        }
        mma_commit_pair(ctl.bar(B_S_FULL + slot));
      };
      // O_slot += P_slot(n) V_n, P read from the slot's S columns
      auto issue_pv = [&](int slot, int n, bool accumulate) {
        const uint64_t dv = smem_desc_sw128(sbase + L::V + (n % kStages) * L::VH, kChunk, 1024);
        const uint32_t tsc = tmem + slot * L::TILE_COLS;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_pair_ts(tsc + 128, tsc + 8 * kk, dv + ((kk * 2048) >> 4), idesc_o, (accumulate || kk > 0));
        mma_commit_pair(ctl.bar(B_O_DONE + slot));
      };
      RunCursor cur(runs), nxt(runs);  // blocks n and n + 1
      bool ok = ctl.wait(B_Q_FULL, 0) && ctl.wait(B_K_FULL, 0);
      if (ok) {
        tc_fence_after();
        if (used(0, cur)) issue_s(0, 0);
        if (used(1, cur)) issue_s(1, 0);
        mma_commit_pair(ctl.bar(B_K_EMPTY));
        if (nblk > 1) nxt.next();
      }
      for (int n = 0; ok && n < nblk; ++n) {
        const int st = n % kStages, st1 = (n + 1) % kStages;
        const bool last = n + 1 == nblk;
        const bool ua = used(0, cur), ub = used(1, cur);
        const bool ua1 = !last && used(0, nxt), ub1 = !last && used(1, nxt);
        if (!last) cur.next();
        if (n + 2 < nblk) nxt.next();
        if (!(ok = ctl.wait(B_V_FULL + st, (n / kStages) & 1))) break;
        if (ua) {
          if (!(ok = ctl.wait_cluster(B_P_FULL, pcount[0] & 1))) break;
          tc_fence_after();
          issue_pv(0, n, pcount[0] > 0);
          ++pcount[0];
        }
        // block n+1's K half: needed from here on
        if (!last && !(ok = ctl.wait(B_K_FULL + st1, ((n + 1) / kStages) & 1))) break;
        tc_fence_after();
        if (ua1) issue_s(0, n + 1);
        if (ub) {
          if (!(ok = ctl.wait_cluster(B_P_FULL + 1, pcount[1] & 1))) break;
          tc_fence_after();
          issue_pv(1, n, pcount[1] > 0);
          ++pcount[1];
        }
        if (ub1) issue_s(1, n + 1);
        if (!last) mma_commit_pair(ctl.bar(B_K_EMPTY + st1));
        mma_commit_pair(ctl.bar(B_V_EMPTY + st));
      }
      mma_commit_pair(ctl.bar(B_MMA_DONE));
      ctl.drain(B_MMA_DONE, 0);
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int slot = warp >> 2;
    const int ti = 2 * slot + int(rank);  // this CTA's tile in the slot
    const bool present = t4[ti] >= 0;
    const int r = threadIdx.x & 127;
    const uint32_t lane_base = uint32_t(32 * (warp & 3)) << 16;
    const uint32_t ts = tmem + slot * L::TILE_COLS + lane_base;  // this row's S (then P) columns; O at +128
    const int q0 = q0s[ti], q1 = q1s[ti];
    const int rows_valid = present ? (q1 - q0) * G : 0;
    const int tok = q0 + r / G;
    const int head = g * G + r % G;
    const float sl2 = s.scale * kLog2e;
    const uint32_t pfull = lead_bar(B_P_FULL + slot);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    uint32_t used = 0;  // blocks this slot has processed
    RunCursor cur(runs);
    for (int n = 0; n < nblk; ++n, cur.next()) {
      if ((cur.end(2 * slot) | cur.end(2 * slot + 1)) == 0) continue;  // the slot does not read this block
      const int kb = cur.kb(), kv1 = cur.end(ti);
      const bool causal = cur.causal(ti);
      if (!(ok = ctl.wait_warp(B_S_FULL + slot, used & 1))) break;
      tc_fence_after();
      if (kv1 == 0) {
        // this CTA's tile does not read the block: P = 0, statistics unchanged
        uint32_t z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) tmem_st16(ts + 16 * c, z);
      } else {
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
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
        const bool full = kb + kBN <= kv1 && (!causal || kb + kBN - 1 <= q0);
        if (!full) {
          const int lim = causal ? min(kv1 - kb, tok - kb + 1) : kv1 - kb;
#pragma unroll
          for (int j = 0; j < kBN; ++j) sv[j] = j < lim ? sv[j] : -INFINITY;
        }
#pragma unroll
        for (int j = 0; j < kBN; j += 2) mx[(j >> 1) & 7] = fmax3(mx[(j >> 1) & 7], sv[j], sv[j + 1]);
        const float mb =
            sl2 * fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        const float m_new = (mb > m_run + kRescaleThreshold) ? mb : m_run;
        const float mref = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = ex2(m_run - mref);
        const float nm = -mref;
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
        // O holds every earlier block of this slot: rescale it in TMEM when a
        // row of the warp needs it
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
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(pfull);
      ++used;
    }
    if (present && ok && used > 0 && ctl.wait_warp(B_O_DONE + slot, (used - 1) & 1)) {
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
  cluster_sync();  // the pair's MMAs are done and neither CTA signals the other any more
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
  clk.end(clk0);
}

}  // namespace

// Launches the paired-SM forward; SP_ERR_UNSUPPORTED when it does not apply
// (head_dim other than 128, or no quads), so the caller can fall back.
int tc_fwd_pair(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, void *o,
                float *lse, int32_t *d_status, void *stream) {
  if (s.D != D || !p.quads || p.n_quads <= 0) return SP_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUtensorMap tq, tk, tv;
  int rc = encode_bf16_3d(&tq, q, D, s.Hq, s.T, 64, s.G, 128 / s.G);
  if (!rc) rc = encode_bf16_3d(&tk, k, D, s.Hkv, s.T, 64, 1, 64);
  if (!rc) rc = encode_bf16_3d(&tv, v, D, s.Hkv, s.T, 64, 1, kBN);
  if (rc) return rc;
  const int smem = Layout::BYTES;
  if (cudaFuncSetAttribute(fwd_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return SP_ERR_CUDA;
  const unsigned grid = 2u * unsigned(p.n_quads) * unsigned(s.Hkv);
  CtaClock clk;
  cta_clock_for(kClockForward, &clk.buf, &clk.cap);
  fwd_pair_kernel<<<grid, kThreads, smem, st>>>(tq, tk, tv, p, s, static_cast<__nv_bfloat16 *>(o), lse, d_status,
                                                clk);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

}  // namespace spc
