// Tree attention forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes: for every query token, softmax attention over the keys of
// its ancestor segments (all visible) and of its own segment up to itself
// (causal), i.e. "causal attention over each query segment's ancestors"
// (PR #7387 "TreePackedSeqParams", "Summary"; issue #7386, "Describe the
// solution you'd like": each query run attends only to its ancestor path).
// Outputs O (bf16) and the natural-log LSE (fp32) kept for the backward.
//
// One CTA per (query tile, KV head).  A tile is 128 rows = (128 / G) tokens x
// the G query heads sharing that KV head, so every K/V block read from L2 or
// HBM feeds a full 128-row MMA even for short segments.  The CTA walks the
// tile's plan ranges in 128-key blocks:
//   warp 4  (one lane)  TMA producer: Q once, then K and V blocks into a
//                       two-stage ring;
//   warp 5  (one lane)  MMA issuer: S = Q K^T into one of two TMEM S buffers,
//                       then O += P V into the TMEM O accumulator, software
//                       pipelined so S of block n+1 runs while the softmax
//                       of block n is computed;
//   warps 0-3           softmax: thread r owns row r (TMEM lane r).  Masks
//                       only where needed (range tail; causal only on blocks
//                       that reach past the tile's first token), online
//                       softmax in the exp2 domain with a lazily updated
//                       reference max (O is rescaled only when the running max
//                       grows by more than 2^8), P rounded to bf16 into
//                       swizzled shared memory, epilogue O / l and LSE.
// Every mbarrier wait is bounded; on expiry the CTA records SP_DEV_TIMEOUT,
// stops issuing work, drains what it issued, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace spc {
namespace {

using namespace ptx;

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per block
constexpr int kStages = 2;        // K/V ring depth
constexpr int kThreads = 192;     // 4 softmax warps + producer + MMA
constexpr int kChunk = 128 * 128; // bytes of one 128-row x 128-byte swizzled chunk
constexpr uint32_t kSpinLimit = 1u << 22;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum : int {
  B_Q_FULL = 0,
  B_K_FULL = 1,   // +stage
  B_K_EMPTY = 3,  // +stage
  B_V_FULL = 5,
  B_V_EMPTY = 7,
  B_S_FULL = 9,   // +buffer
  B_S_FREE = 11,  // +buffer
  B_P_FULL = 13,
  B_PV_DONE = 14,
  B_MMA_DONE = 15,
  B_COUNT = 16
};

template <int D>
struct Layout {
  static constexpr int kDChunks = D / 64;
  static constexpr int Q = 0;
  static constexpr int KV = kDChunks * kChunk;  // bytes of 128 rows x D
  static constexpr int K = Q + KV;
  static constexpr int V = K + kStages * KV;
  static constexpr int P = V + kStages * KV;
  static constexpr int BAR = P + 2 * kChunk;
  static constexpr int TSLOT = BAR + 8 * B_COUNT;
  static constexpr int ABORT = TSLOT + 4;
  static constexpr int BYTES = ABORT + 4 + 1024;  // + alignment slack
  // at least ~116 KB so two CTAs never share an SM (each takes all 512 TMEM columns)
  static constexpr int ALLOC = BYTES > 120 * 1024 ? BYTES : 120 * 1024;
};

struct Ctl {
  uint32_t bar0;
  volatile int *abort;
  int32_t *d_status;
  __device__ uint32_t bar(int i) const { return bar0 + 8u * uint32_t(i); }
  // Bounded wait; false if it expired here or another role gave up first.
  __device__ bool wait(int i, uint32_t parity) const {
    for (uint32_t it = 0;; ++it) {
      if (mbar_try_wait(bar(i), parity)) return true;
      if ((it & 255u) == 255u) {
        if (*abort) return false;
        if (it >= kSpinLimit) {
          *abort = 1;
          if (d_status) atomicOr(d_status, SP_DEV_TIMEOUT);
          return false;
        }
      }
    }
  }
  // Bounded wait used while draining after an abort (ignores the flag).
  // Same for a whole warp: one lane polls (32 lanes polling one barrier
  // serialise on it and starve the warps that do the work), the others wait
  // at __syncwarp, which also orders their later reads after lane 0's acquire.
  __device__ bool wait_warp(int i, uint32_t parity) const {
    bool r = true;
    if ((threadIdx.x & 31) == 0) r = wait(i, parity);
    __syncwarp();
    return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
  }
  __device__ void drain(int i, uint32_t parity) const {
    for (uint32_t it = 0; it < kSpinLimit; ++it)
      if (mbar_try_wait(bar(i), parity)) return;
  }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, PlanDev plan, AttnShape s,
                  __nv_bfloat16 *__restrict__ o, float *__restrict__ lse, int32_t *d_status) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived by pointer arithmetic so that accesses
  // through it stay shared-memory (not generic) accesses
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int g = blockIdx.x / plan.n_tiles;
  const int *tile = plan.tiles + 5 * (blockIdx.x % plan.n_tiles);
  const int q0 = tile[1], q1 = tile[2], rb = tile[3], rc = tile[4];
  const int G = s.G, T = s.T;
  const int *rng = plan.ranges + 2 * rb;

  // Validate the work item (uniform over the CTA) and count its key blocks.
  bool bad = !(0 <= q0 && q0 < q1 && q1 <= T && rc >= 1);
  int nblocks = 0;
  for (int i = 0; !bad && i < rc; ++i) {
    const int a = rng[2 * i], b = rng[2 * i + 1];
    if (!(0 <= a && a < b && b <= T)) bad = true;
    nblocks += (b - a + kBN - 1) / kBN;
  }
  if (bad) {
    if (threadIdx.x == 0 && d_status) atomicOr(d_status, SP_DEV_BAD_PLAN);
    return;
  }

  Ctl ctl{sbase + L::BAR, reinterpret_cast<volatile int *>(smem + L::ABORT), d_status};
  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      const uint32_t cnt = (i == B_S_FREE || i == B_S_FREE + 1 || i == B_P_FULL) ? 128u : 1u;
      mbar_init(ctl.bar(i), cnt);
    }
    *ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(sbase + L::TSLOT, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::TSLOT);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(ctl.bar(B_Q_FULL), L::KV);
#pragma unroll
      for (int c = 0; c < L::kDChunks; ++c)
        tma_load_3d(sbase + L::Q + c * kChunk, &tm_q, ctl.bar(B_Q_FULL), c * 64, g * G, q0);
      int n = 0;
      bool ok = true;
      for (int ri = 0; ok && ri < rc; ++ri) {
        const int kv0 = rng[2 * ri], kv1 = rng[2 * ri + 1];
        for (int kb = kv0; kb < kv1; kb += kBN, ++n) {
          const int st = n & 1;
          const uint32_t ph = (n >> 1) & 1;
          if (!(ok = ctl.wait(B_K_EMPTY + st, ph ^ 1))) break;
          mbar_arrive_expect_tx(ctl.bar(B_K_FULL + st), L::KV);
#pragma unroll
          for (int c = 0; c < L::kDChunks; ++c)
            tma_load_3d(sbase + L::K + st * L::KV + c * kChunk, &tm_k, ctl.bar(B_K_FULL + st), c * 64, g, kb);
          if (!(ok = ctl.wait(B_V_EMPTY + st, ph ^ 1))) {
            ctl.drain(B_K_FULL + st, ph);
            break;
          }
          mbar_arrive_expect_tx(ctl.bar(B_V_FULL + st), L::KV);
#pragma unroll
          for (int c = 0; c < L::kDChunks; ++c)
            tma_load_3d(sbase + L::V + st * L::KV + c * kChunk, &tm_v, ctl.bar(B_V_FULL + st), c * 64, g, kb);
        }
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
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, 0, 1);
      const uint32_t tO = tmem + 256;
      // operand descriptors, built once; a K step only moves the start address
      const uint64_t dq0 = smem_desc_sw128(sbase + L::Q, 16, 1024);
      const uint64_t dk_s0 = smem_desc_sw128(sbase + L::K, 16, 1024);
      const uint64_t dk_s1 = smem_desc_sw128(sbase + L::K + L::KV, 16, 1024);
      const uint64_t dp0 = smem_desc_sw128(sbase + L::P, 16, 1024);
      const uint64_t dv_s0 = smem_desc_sw128(sbase + L::V, kChunk, 1024);
      const uint64_t dv_s1 = smem_desc_sw128(sbase + L::V + L::KV, kChunk, 1024);
      if (ctl.wait(B_Q_FULL, 0)) {
        tc_fence_after();
        for (int n = 0; n <= nblocks; ++n) {
          if (n < nblocks) {
            const int st = n & 1;
            const uint32_t ph = (n >> 1) & 1;
            if (!ctl.wait(B_K_FULL + st, ph)) break;
            if (!ctl.wait(B_S_FREE + st, ph ^ 1)) break;
            tc_fence_after();
            const uint64_t dk = st ? dk_s1 : dk_s0;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
              mma_bf16_ss(tmem + st * 128, dq0 + off, dk + off, idesc_s, kk > 0);
            }
            mma_commit(ctl.bar(B_S_FULL + st));
            mma_commit(ctl.bar(B_K_EMPTY + st));
          }
          if (n >= 1) {
            const int m = n - 1, st = m & 1;
            const uint32_t ph = (m >> 1) & 1;
            if (!ctl.wait(B_P_FULL, m & 1)) break;
            if (!ctl.wait(B_V_FULL + st, ph)) break;
            tc_fence_after();
            const uint64_t dv = st ? dv_s1 : dv_s0;
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk) {
              const uint32_t poff = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
              mma_bf16_ss(tO, dp0 + poff, dv + ((kk * 2048) >> 4), idesc_o, (m > 0 || kk > 0));
            }
            mma_commit(ctl.bar(B_V_EMPTY + st));
            mma_commit(ctl.bar(B_PV_DONE));
          }
        }
      }
      mma_commit(ctl.bar(B_MMA_DONE));
      ctl.drain(B_MMA_DONE, 0);
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int r = threadIdx.x;
    const uint32_t lane_base = uint32_t(32 * warp) << 16;
    const int rows_valid = (q1 - q0) * G;
    const int tok = q0 + r / G;
    const int head = g * G + r % G;
    const float sl2 = s.scale * kLog2e;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int n = 0;
    const uint32_t prow = sbase + L::P + r * 128;
    for (int ri = 0; ok && ri < rc; ++ri) {
      const int kv0 = rng[2 * ri], kv1 = rng[2 * ri + 1];
      const bool causal = ri == rc - 1;
      for (int kb = kv0; kb < kv1; kb += kBN, ++n) {
        const int sb = n & 1;
        if (!(ok = ctl.wait_warp(B_S_FULL + sb, (n >> 1) & 1))) break;
        tc_fence_after();
        float sv[kBN];
#pragma unroll
        for (int c = 0; c < kBN / 64; ++c) {
          uint32_t u0[32], u1[32];
          tmem_ld32x2(tmem + lane_base + sb * 128 + 64 * c, tmem + lane_base + sb * 128 + 64 * c + 32, u0, u1);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            sv[64 * c + j] = __uint_as_float(u0[j]);
            sv[64 * c + 32 + j] = __uint_as_float(u1[j]);
          }
        }
        tc_fence_before();
        mbar_arrive(ctl.bar(B_S_FREE + sb));

        // scale (and mask) in the log2 domain; row max by a tree of 8 partials
        float mx[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) mx[t] = -INFINITY;
        if (kb + kBN <= kv1 && (!causal || kb + kBN - 1 <= q0)) {
#pragma unroll
          for (int j = 0; j < kBN; ++j) {
            sv[j] *= sl2;
            mx[j & 7] = fmaxf(mx[j & 7], sv[j]);
          }
        } else {
          const int lim = causal ? min(kv1 - kb, tok - kb + 1) : kv1 - kb;
#pragma unroll
          for (int j = 0; j < kBN; ++j) {
            sv[j] = j < lim ? sv[j] * sl2 : -INFINITY;
            mx[j & 7] = fmaxf(mx[j & 7], sv[j]);
          }
        }
        const float mb = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float m_new = (mb > m_run + kRescaleThreshold) ? mb : m_run;
        const float mref = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = ex2(m_run - mref);
        // subtract, then all exponentials back to back, then a tree sum
#pragma unroll
        for (int j = 0; j < kBN; ++j) sv[j] -= mref;
#pragma unroll
        for (int j = 0; j < kBN; ++j) sv[j] = ex2(sv[j]);
        float sm[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) sm[t] = 0.f;
#pragma unroll
        for (int j = 0; j < kBN; ++j) sm[j & 7] += sv[j];
        const float rs = ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
        l_run = l_run * alpha + rs;

        if (n >= 1) {
          if (!(ok = ctl.wait_warp(B_PV_DONE, (n - 1) & 1))) break;
          tc_fence_after();
        }
        // P row -> shared memory, bf16, K-major with the 128-byte swizzle
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float *x = sv + 64 * c + 8 * j;
            st_shared_v4(prow + c * kChunk + ((j ^ (r & 7)) << 4), pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]),
                         pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
          }
        }
        if (n >= 1) {
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            const uint32_t ta = tmem + lane_base + 256;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {  // 64 columns at a time
              uint32_t u0[32], u1[32];
              tmem_ld32x2(ta + 64 * c, ta + 64 * c + 32, u0, u1);
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                u0[j] = __float_as_uint(__uint_as_float(u0[j]) * alpha);
                u1[j] = __float_as_uint(__uint_as_float(u1[j]) * alpha);
              }
              tmem_st32(ta + 64 * c, u0);
              tmem_st32(ta + 64 * c + 32, u1);
            }
            tmem_st_wait();
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(ctl.bar(B_P_FULL));
        m_run = m_new;
      }
    }
    if (ok && ctl.wait_warp(B_PV_DONE, (nblocks - 1) & 1)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const bool store = r < rows_valid;
      __nv_bfloat16 *orow = o + (size_t(tok) * s.Hq + head) * D;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t u0[32], u1[32];
        tmem_ld32x2(tmem + lane_base + 256 + 64 * c, tmem + lane_base + 256 + 64 * c + 32, u0, u1);
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
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
int launch(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, void *o, float *lse,
           int32_t *d_status, cudaStream_t st) {
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
  const unsigned grid = unsigned(p.n_tiles) * unsigned(s.Hkv);
  kern<<<grid, kThreads, smem, st>>>(tq, tk, tv, p, s, static_cast<__nv_bfloat16 *>(o), lse, d_status);
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
