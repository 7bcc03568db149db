// Deterministic dQ of shared-prefix tree attention: each query tile walks
// its own ancestor key ranges ("[ENHANCEMENT] Shared-prefix training with
// context parallelism for exact agent trajectories", issue #7386, "Describe
// the solution you'd like": each query run attends to its ancestor path; PR
// #7387 "TreePackedSeqParams", "Summary": a query segment attends causally
// over its ancestors) and accumulates
//
//   dQ = scale * sum_keys dS K,   dS = P o (dP - Delta),  P = exp(scale Q K^T - LSE),  dP = dO V^T
//
// in TMEM, in the plan's fixed block order, so dQ is the same bit for bit on
// every run (the atomic path adds key blocks' partials in arrival order).
//
// dq_tc_kernel: one CTA per (128-row query tile, KV head), KV head outermost
// so a head's K/V stays in L2 while its tiles run.  Warps 0-7: elementwise,
// thread = query row = TMEM lane, warpgroup h taking key columns
// [64h, 64h + 64) of every row (the work needs no row reduction, so the
// split needs no exchange); warp 8: TMA producer (Q and dO once, K/V blocks
// through rings of three and two stages: K is read last by dQ, V only by
// dP, so a third K stage gives the next blocks' loads time to land); warps 9
// and 10: one tcgen05 MMA issuer each.  Per key block n warp 9 issues
// S = Q K^T and dP = dO V^T (SS), and warp 10, once the elementwise warps
// have stored dS(n) as bf16 pairs in TMEM, dQ += dS(n) K(n) (A read from
// TMEM, K as an MN-major B).  The two issuers share the tensor pipe but wait
// on their own barriers: an mbarrier wait costs the waiting thread about a
// hundred cycles even when the phase is already complete, and a thread
// blocked there issues nothing, so one issuer's waits run while the other's
// products keep the pipe busy.  Their products touch disjoint TMEM columns
// and every hand-over between them goes through the elementwise warps'
// barriers, so no ordering between the two threads' products is needed.  S(n+1) is issued as soon as S(n)
// has been read and dP(n+1) as soon as dP(n) has, so both run while dS(n) is
// formed; the elementwise warps read S, release it, take the exponentials,
// then read and release dP.  dS alternates between two TMEM buffers.
// TMEM: S 128 + dP 128 + dQ D + 2 x 64 (dS) <= 512 columns.
//
// Every wait is bounded (Ctl): on expiry the CTA sets SP_DEV_TIMEOUT, stops
// issuing, drains its copies and MMAs, frees TMEM and returns.
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

constexpr int kBM = 128;           // query rows per tile (tokens x query heads of one KV head)
constexpr int kBN = 128;           // keys per block
constexpr int kKStages = 3;        // K ring depth (K is read by S and, last, by dQ)
constexpr int kVStages = 2;        // V ring depth (V is read by dP only)
constexpr int kThreads = 352;      // 8 elementwise warps, producer, two MMA issuers
constexpr int kChunk = 128 * 128;  // one 128-row x 128-byte swizzled chunk
constexpr float kLog2e = 1.4426950408889634f;

enum : int {
  B_Q_FULL = 0,
  B_K_FULL = 1,    // +stage (3)
  B_K_EMPTY = 4,   // +stage
  B_V_FULL = 7,    // +stage (2)
  B_V_EMPTY = 9,   // +stage
  B_S_FULL = 11,
  B_DP_FULL = 12,
  B_S_FREE = 13,   // 8 warp arrivals
  B_DP_FREE = 14,  // 8 warp arrivals
  B_DS_FULL = 15,  // +buffer, 8 warp arrivals
  B_DS_FREE = 17,  // +buffer
  B_DQ_DONE = 19,
  B_SDP_DONE = 20,  // the S / dP issuer's last products have completed
  B_COUNT = 21
};

template <int D>
struct Layout {
  static constexpr int kDChunks = D / 64;
  static constexpr int KV = kDChunks * kChunk;  // bytes of 128 rows x D
  static constexpr int Q = 0;
  static constexpr int DO = KV;
  static constexpr int K = 2 * KV;  // + stage * KV
  static constexpr int V = K + kKStages * KV;
  static constexpr int BAR = V + kVStages * KV;
  static constexpr int TSLOT = BAR + 8 * B_COUNT;
  static constexpr int ABORT = TSLOT + 4;
  static constexpr int BYTES = ABORT + 4 + 1024;
  // at least ~116 KB so two CTAs never share an SM (each takes all 512 TMEM columns)
  static constexpr int ALLOC = BYTES > 120 * 1024 ? BYTES : 120 * 1024;
};

constexpr uint32_t T_S = 0, T_DP = 128, T_DQ = 256, T_DS = 384;

// Walks a tile's key blocks: ranges in plan order, 128 keys at a time.
struct BlockWalk {
  const int *rg;
  int rc, r, kb;
  __device__ BlockWalk(const int *ranges, int count) : rg(ranges), rc(count), r(0), kb(ranges[0]) {}
  __device__ int end() const { return rg[2 * r + 1]; }
  __device__ bool causal() const { return r == rc - 1; }
  __device__ void next() {
    kb += kBN;
    if (kb >= rg[2 * r + 1] && ++r < rc) kb = rg[2 * r];
  }
};

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, PlanDev plan,
                 AttnShape s, const float *__restrict__ lse, const float *__restrict__ delta,
                 __nv_bfloat16 *__restrict__ dq, int32_t *d_status, CtaClock clk) {
  using L = Layout<D>;
  const unsigned long long clk0 = clk.begin();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = s.T;

  const int g = blockIdx.x / plan.n_tiles;
  const int *tl = plan.tiles + 5 * (blockIdx.x % plan.n_tiles);
  const int q0 = tl[1], q1 = tl[2], rb = tl[3], rc = tl[4];
  const int *rg = plan.ranges + 2 * rb;
  // Validate the work item (uniform over the CTA) and count its key blocks.
  bool bad = !(0 <= q0 && q0 < q1 && q1 <= T && (q1 - q0) * G <= kBM && rc >= 1);
  int nblk = 0;
  for (int i = 0; !bad && i < rc; ++i) {
    const int a = rg[2 * i], e = rg[2 * i + 1];
    if (!(0 <= a && a < e && e <= T)) bad = true;
    nblk += (e - a + kBN - 1) / kBN;
  }
  if (bad) {
    if (threadIdx.x == 0 && d_status) atomicOr(d_status, SP_DEV_BAD_PLAN);
    return;
  }

  Ctl ctl{sbase + L::BAR, reinterpret_cast<volatile int *>(smem + L::ABORT), d_status, kSpinLimit};
  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(ctl.bar(i), (i == B_S_FREE || i == B_DP_FREE || i == B_DS_FULL || i == B_DS_FULL + 1) ? 8u : 1u);
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
      mbar_arrive_expect_tx(ctl.bar(B_Q_FULL), 2u * L::KV);
#pragma unroll
      for (int c = 0; c < L::kDChunks; ++c) {
        tma_load_3d(sbase + L::Q + c * kChunk, &tm_q, ctl.bar(B_Q_FULL), c * 64, g * G, q0);
        tma_load_3d(sbase + L::DO + c * kChunk, &tm_do, ctl.bar(B_Q_FULL), c * 64, g * G, q0);
      }
      BlockWalk w(rg, rc);
      int nk = 0, nv = 0;  // K and V blocks issued
      for (int n = 0; n < nblk; ++n, w.next()) {
        const int ks = n % kKStages, vs = n % kVStages;
        if (!ctl.wait(B_K_EMPTY + ks, ((n / kKStages) & 1) ^ 1)) break;
        mbar_arrive_expect_tx(ctl.bar(B_K_FULL + ks), L::KV);
#pragma unroll
        for (int c = 0; c < L::kDChunks; ++c)
          tma_load_3d(sbase + L::K + ks * L::KV + c * kChunk, &tm_k, ctl.bar(B_K_FULL + ks), c * 64, g, w.kb);
        ++nk;
        if (!ctl.wait(B_V_EMPTY + vs, ((n / kVStages) & 1) ^ 1)) break;
        mbar_arrive_expect_tx(ctl.bar(B_V_FULL + vs), L::KV);
#pragma unroll
        for (int c = 0; c < L::kDChunks; ++c)
          tma_load_3d(sbase + L::V + vs * L::KV + c * kChunk, &tm_v, ctl.bar(B_V_FULL + vs), c * 64, g, w.kb);
        ++nv;
      }
      if (*ctl.abort) {
        // let the fills still in flight land before the CTA exits
        ctl.drain(B_Q_FULL, 0);
        for (int m = nk - kKStages < 0 ? 0 : nk - kKStages; m < nk; ++m)
          ctl.drain(B_K_FULL + m % kKStages, (m / kKStages) & 1);
        for (int m = nv - kVStages < 0 ? 0 : nv - kVStages; m < nv; ++m)
          ctl.drain(B_V_FULL + m % kVStages, (m / kVStages) & 1);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------- S and dP MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(kBM, kBN, 0, 0);  // S = Q K^T, dP = dO V^T
      const uint64_t dq_a = smem_desc_sw128(sbase + L::Q, 16, 1024);
      const uint64_t ddo_a = smem_desc_sw128(sbase + L::DO, 16, 1024);
      // S(n) = Q K(n)^T into TMEM
      auto issue_s = [&](int n) {
        const uint64_t dk = smem_desc_sw128(sbase + L::K + (n % kKStages) * L::KV, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + T_S, dq_a + off, dk + off, id_s, kk > 0);
        }
        mma_commit(ctl.bar(B_S_FULL));
      };
      // dP(n) = dO V(n)^T into TMEM
      auto issue_dp = [&](int n) {
        const uint64_t dv = smem_desc_sw128(sbase + L::V + (n % kVStages) * L::KV, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + T_DP, ddo_a + off, dv + off, id_s, kk > 0);
        }
        mma_commit(ctl.bar(B_DP_FULL));
        mma_commit(ctl.bar(B_V_EMPTY + n % kVStages));  // V(n) is read by dP(n) only
      };
      bool ok = ctl.wait(B_Q_FULL, 0) && ctl.wait(B_K_FULL, 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      if (ok && (ok = ctl.wait(B_V_FULL, 0))) {
        tc_fence_after();
        issue_dp(0);
      }
      for (int n = 0; ok && n + 1 < nblk; ++n) {
        {
          // S(n) has been read out: S(n+1) may overwrite it; likewise dP
          if (!(ok = ctl.wait(B_S_FREE, n & 1))) break;
          if (!(ok = ctl.wait(B_K_FULL + (n + 1) % kKStages, ((n + 1) / kKStages) & 1))) break;
          tc_fence_after();
          issue_s(n + 1);
          if (!(ok = ctl.wait(B_DP_FREE, n & 1))) break;
          if (!(ok = ctl.wait(B_V_FULL + (n + 1) % kVStages, ((n + 1) / kVStages) & 1))) break;
          tc_fence_after();
          issue_dp(n + 1);
        }
      }
      // every S and dP product of this thread has completed before TMEM is freed
      mma_commit(ctl.bar(B_SDP_DONE));
      ctl.drain(B_SDP_DONE, 0);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------ dQ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_q = idesc_bf16_f32(kBM, D, 0, 1);  // dQ += dS K (K as MN-major B)
      bool ok = true;
      for (int n = 0; ok && n < nblk; ++n) {
        const int st = n & 1;
        // dS(n) in TMEM (so S(n), and the K(n) it read, are complete); K(n) still checked
        if (!(ok = ctl.wait(B_DS_FULL + st, (n >> 1) & 1))) break;
        if (!(ok = ctl.wait(B_K_FULL + n % kKStages, (n / kKStages) & 1))) break;
        tc_fence_after();
        const uint64_t dk_mn = smem_desc_sw128(sbase + L::K + (n % kKStages) * L::KV, kChunk, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_bf16_ts(tmem + T_DQ, tmem + T_DS + 64 * st + 8 * kk, dk_mn + ((kk * 2048) >> 4), id_q,
                      (n > 0 || kk > 0));
        mma_commit(ctl.bar(B_DS_FREE + st));
        mma_commit(ctl.bar(B_K_EMPTY + n % kKStages));  // S(n) read K(n) before dS(n) existed
      }
      mma_commit(ctl.bar(B_DQ_DONE));
      ctl.drain(B_DQ_DONE, 0);
    }
  } else {
    // --------------------------------------------------------- elementwise
    const int h = warp >> 2;            // key columns [64h, 64h + 64)
    const int r = threadIdx.x & 127;    // query row = TMEM lane
    const uint32_t lane_base = uint32_t(32 * (warp & 3)) << 16;
    const int tok = q0 + r / G, head = g * G + r % G;
    const bool rowv = tok < q1;
    const float sl2 = s.scale * kLog2e;
    const float nl2 = rowv ? -__ldg(lse + size_t(head) * T + tok) * kLog2e : 0.f;
    const float ndl = rowv ? -__ldg(delta + size_t(head) * T + tok) : 0.f;
    BlockWalk w(rg, rc);
    bool ok = true;
    for (int n = 0; n < nblk; ++n, w.next()) {
      const int st = n & 1;
      if (!(ok = ctl.wait_warp(B_S_FULL, n & 1))) break;
      tc_fence_after();
      const int kv1 = w.end(), kb = w.kb;
      const bool causal = w.causal();
      // every row of the tile sees every key of the block
      const bool full = kb + kBN <= kv1 && (!causal || kb + kBN - 1 <= q0);
      // keys [kb, kb + lim) visible to this row
      const int lim = !rowv ? 0 : (causal ? min(kv1 - kb, tok - kb + 1) : kv1 - kb);
      // this group's 64 columns of S, all loaded before S_FREE so the next
      // block's S product can start at once
      uint32_t us[64], ud[64];
      tmem_ld32x2(tmem + lane_base + T_S + 64 * h, tmem + lane_base + T_S + 64 * h + 32,
                  *reinterpret_cast<uint32_t(*)[32]>(us), *reinterpret_cast<uint32_t(*)[32]>(us + 32));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ctl.bar(B_S_FREE));
      // P (in place of S), then dS (in place of dP)
      if (full && rowv) {
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          float p0, p1;
          ffma2(p0, p1, __uint_as_float(us[i]), __uint_as_float(us[i + 1]), sl2, sl2, nl2, nl2);
          us[i] = __float_as_uint(p0), us[i + 1] = __float_as_uint(p1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          us[i] = __float_as_uint(64 * h + i < lim ? fmaf(__uint_as_float(us[i]), sl2, nl2) : -INFINITY);
      }
#pragma unroll
      for (int i = 0; i < 64; ++i) us[i] = __float_as_uint(ex2(__uint_as_float(us[i])));
      // this group's 64 columns of dP, released as soon as they are read
      if (!(ok = ctl.wait_warp(B_DP_FULL, n & 1))) break;
      tc_fence_after();
      tmem_ld32x2(tmem + lane_base + T_DP + 64 * h, tmem + lane_base + T_DP + 64 * h + 32,
                  *reinterpret_cast<uint32_t(*)[32]>(ud), *reinterpret_cast<uint32_t(*)[32]>(ud + 32));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ctl.bar(B_DP_FREE));
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        float t0, t1, d0, d1;
        fadd2(t0, t1, __uint_as_float(ud[i]), __uint_as_float(ud[i + 1]), ndl, ndl);
        fmul2(d0, d1, __uint_as_float(us[i]), __uint_as_float(us[i + 1]), t0, t1);
        pk[i / 2] = pack_bf16(d0, d1);
      }
      // dS(n) goes to buffer st once dQ(n-2) has read it
      if (!(ok = ctl.wait_warp(B_DS_FREE + st, ((n >> 1) & 1) ^ 1))) break;
      tmem_st32(tmem + lane_base + T_DS + 64 * st + 32 * h, pk);
      if (!ok) break;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ctl.bar(B_DS_FULL + st));
    }
    if (ok && ctl.wait_warp(B_DQ_DONE, 0)) {
      tc_fence_after();
      __nv_bfloat16 *row = dq + (size_t(tok) * s.Hq + head) * D;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {  // head-dim columns [D/2 h, D/2 (h + 1))
        const int c = (D / 64) * h + cc;
        uint32_t u[32];
        tmem_ld32(tmem + lane_base + T_DQ + 32 * c, u);
        if (rowv) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(u[i]) * s.scale, __uint_as_float(u[i + 1]) * s.scale);
            v.y = pack_bf16(__uint_as_float(u[i + 2]) * s.scale, __uint_as_float(u[i + 3]) * s.scale);
            v.z = pack_bf16(__uint_as_float(u[i + 4]) * s.scale, __uint_as_float(u[i + 5]) * s.scale);
            v.w = pack_bf16(__uint_as_float(u[i + 6]) * s.scale, __uint_as_float(u[i + 7]) * s.scale);
            *reinterpret_cast<uint4 *>(row + 32 * c + i) = v;
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
           const void *d_o, void *dq, const float *delta, int32_t *d_status, cudaStream_t st) {
  CUtensorMap tq, tdo, tk, tv;
  int rc = encode_bf16_3d(&tq, q, D, s.Hq, s.T, 64, G, kBM / G);
  if (!rc) rc = encode_bf16_3d(&tdo, d_o, D, s.Hq, s.T, 64, G, kBM / G);
  if (!rc) rc = encode_bf16_3d(&tk, k, D, s.Hkv, s.T, 64, 1, kBN);
  if (!rc) rc = encode_bf16_3d(&tv, v, D, s.Hkv, s.T, 64, 1, kBN);
  if (rc) return rc;
  auto kern = dq_tc_kernel<D, G>;
  const int smem = Layout<D>::ALLOC;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return SP_ERR_CUDA;
  const unsigned grid = unsigned(p.n_tiles) * unsigned(s.Hkv);
  CtaClock clk;
  cta_clock_for(kClockQueryTiles, &clk.buf, &clk.cap);
  kern<<<grid, kThreads, smem, st>>>(tq, tdo, tk, tv, p, s, lse, delta, static_cast<__nv_bfloat16 *>(dq), d_status,
                                     clk);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

}  // namespace

int tc_dq(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, const float *lse,
          const void *d_o, void *dq, const float *delta, int32_t *d_status, void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
#define SPC_DQ_CASE(DD, GG) \
  if (s.D == DD && s.G == GG) return launch<DD, GG>(p, s, q, k, v, lse, d_o, dq, delta, d_status, st);
  SPC_DQ_CASE(64, 1) SPC_DQ_CASE(64, 2) SPC_DQ_CASE(64, 4) SPC_DQ_CASE(64, 8)
  SPC_DQ_CASE(128, 1) SPC_DQ_CASE(128, 2) SPC_DQ_CASE(128, 4) SPC_DQ_CASE(128, 8)
#undef SPC_DQ_CASE
  return SP_ERR_UNSUPPORTED;
}

}  // namespace spc
