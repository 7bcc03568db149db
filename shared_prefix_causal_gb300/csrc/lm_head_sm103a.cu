// Vocabulary head over the sampled-edge states: per-action log-probability of
// the sampled token ("[ENHANCEMENT] Shared-prefix training with context
// parallelism for exact agent trajectories", issue #7386, "Describe the
// solution you'd like", fifth bullet: only sampled-edge source states are
// projected, a single loss owner for each sampled action; "TreePackedSeqParams" draft,
// PR #7387, "Summary": edge-source selection before the vocabulary projection).
//
//   logits[e][v] = <h[e], W[v]>    (h: [E][Hd], W: [V][Hd], bf16; fp32 accumulation)
//   lse[e]       = log sum_v exp(logits[e][v])
//   logprob[e]   = logits[e][labels[e]] - lse[e]
//
// and, for an upstream gradient g[e] = dL/dlogprob[e],
//
//   dlogits[e][v] = g[e] * (1[v == labels[e]] - exp(logits[e][v] - lse[e]))
//   d_hidden_sel  = dlogits W,    d_weight = dlogits^T h
//
// gemm_kernel: persistent tcgen05 GEMM over 128 x 256 output tiles.  A 4-stage
// TMA ring feeds 128x256x16 MMAs into one of two 256-column TMEM accumulators
// while the epilogue warpgroup (thread = output row = TMEM lane) drains the
// other.  Operands are K-major or MN-major (128-byte swizzle either way), so
// all four products read the row-major tensors as they are.  Epilogues:
//   LseEpi      forward: per tile the row maximum, the sum of exponentials and
//               the label's logit; the [E][V] logits never reach memory, and
//               lmh_combine_kernel merges the tile partials into lse, logprob.
//   DlogitsEpi  backward: recomputed logits -> bf16 dlogits [E][V].
//   StoreEpi    fp32 store (d_hidden_sel, d_weight).
// Vocabulary blocks are the outer tile loop for the projections, so CTAs
// running side by side read the same W block while h stays in L2; for
// d_weight the hidden blocks of one vocabulary block run side by side.
//
// Every mbarrier wait is bounded (Ctl): on expiry the CTA sets SP_DEV_TIMEOUT,
// stops issuing, lets its copies and MMAs finish, frees TMEM and returns.
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

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kThreads = 256;  // warp 0 TMA, warp 1 MMA + TMEM owner, warps 4-7 epilogue
constexpr uint32_t kABytes = kBM * kBK * 2, kBBytes = kBN * kBK * 2, kStage = kABytes + kBBytes;
constexpr float kL2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;

enum : int {
  B_FULL = 0,                   // [kStages] TMA -> MMA
  B_EMPTY = kStages,            // [kStages] MMA -> TMA
  B_ACC_FULL = 2 * kStages,     // [2] MMA -> epilogue
  B_ACC_EMPTY = 2 * kStages + 2,  // [2] epilogue (4 warps) -> MMA
  B_DONE = 2 * kStages + 4,     // last MMA of the CTA complete
  B_COUNT
};
constexpr uint32_t SM_BAR = kStages * kStage;
constexpr uint32_t SM_ABORT = SM_BAR + 8 * B_COUNT;
constexpr uint32_t SM_TSLOT = SM_ABORT + 8;
constexpr uint32_t SM_ALLOC = SM_TSLOT + 8 + 1024;  // + slack for the 1024-byte alignment

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Persistent GEMM D[M][N] = sum_k A[m][k] B[n][k] in 128 x 256 tiles.  A is
// K-major (A[m][k] at a + m*K + k) or MN-major (at a + k*M + m); the same for
// B.  Epi consumes each finished accumulator.
struct GemmShape {
  int32_t M, N, K;
  int32_t m_tiles, n_tiles, k_blocks;
  int32_t m_fast;  // tile order: 1 = m varies fastest, 0 = n varies fastest
  __device__ __forceinline__ void tile(int t, int &m0, int &n0) const {
    if (m_fast) {
      m0 = (t % m_tiles) * kBM;
      n0 = (t / m_tiles) * kBN;
    } else {
      n0 = (t % n_tiles) * kBN;
      m0 = (t / n_tiles) * kBM;
    }
  }
};

// Shared-memory tile layouts (128-byte swizzle).  K-major: rows of 64 K values
// (128 bytes), 8-row atoms 1024 bytes apart; a 16-wide K step moves the start
// by 32 bytes.  MN-major: per 64-wide M/N block, 64 rows along K of 128 bytes
// (8 KB), blocks 8 KB apart; a 16-wide K step moves the start by 2048 bytes.
constexpr uint32_t kMnBlock = 64 * 128;

template <bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, GemmShape s,
                Epi epi, int32_t *d_status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles_total = s.m_tiles * s.n_tiles;

  Ctl ctl{sbase + SM_BAR, reinterpret_cast<volatile int *>(smem + SM_ABORT), d_status, kSpinLimit};
  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(ctl.bar(i), (i == B_ACC_EMPTY || i == B_ACC_EMPTY + 1) ? 4u : 1u);
    *ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + SM_TSLOT, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + SM_TSLOT);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_a);
      prefetch_tmap(&tm_b);
      uint32_t it = 0;  // stage fills issued
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles_total; t += gridDim.x) {
        int m0, n0;
        s.tile(t, m0, n0);
        for (int kb = 0; kb < s.k_blocks; ++kb, ++it) {
          const uint32_t st = it % kStages, ph = (it / kStages) & 1;
          if (!(ok = ctl.wait(B_EMPTY + st, ph ^ 1))) break;
          const uint32_t dst = sbase + st * kStage, bar = ctl.bar(B_FULL + st);
          mbar_arrive_expect_tx(bar, kStage);
          if constexpr (A_MN) {
#pragma unroll
            for (int j = 0; j < kBM / 64; ++j) tma_load_2d(dst + j * kMnBlock, &tm_a, bar, m0 + 64 * j, kb * kBK);
          } else {
            tma_load_2d(dst, &tm_a, bar, kb * kBK, m0);
          }
          if constexpr (B_MN) {
#pragma unroll
            for (int j = 0; j < kBN / 64; ++j)
              tma_load_2d(dst + kABytes + j * kMnBlock, &tm_b, bar, n0 + 64 * j, kb * kBK);
          } else {
            tma_load_2d(dst + kABytes, &tm_b, bar, kb * kBK, n0);
          }
        }
      }
      if (!ok) {
        // let the fills still in flight land before the CTA exits
        for (uint32_t j = it > kStages ? it - kStages : 0; j < it; ++j)
          ctl.drain(B_FULL + j % kStages, (j / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, A_MN ? 1 : 0, B_MN ? 1 : 0);
      constexpr uint32_t a_lbo = A_MN ? kMnBlock : 16, b_lbo = B_MN ? kMnBlock : 16;
      constexpr uint32_t a_step = A_MN ? (16 * 128) >> 4 : 32 >> 4, b_step = B_MN ? (16 * 128) >> 4 : 32 >> 4;
      uint32_t it = 0, lt = 0;  // stages consumed, tiles issued
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles_total; t += gridDim.x, ++lt) {
        const uint32_t acc = lt & 1;
        if (!(ok = ctl.wait(B_ACC_EMPTY + acc, ((lt >> 1) & 1) ^ 1))) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * kBN;
        for (int kb = 0; kb < s.k_blocks; ++kb, ++it) {
          const uint32_t st = it % kStages, ph = (it / kStages) & 1;
          if (!(ok = ctl.wait(B_FULL + st, ph))) break;
          tc_fence_after();
          const uint64_t da = smem_desc_sw128(sbase + st * kStage, a_lbo, 1024);
          const uint64_t db = smem_desc_sw128(sbase + st * kStage + kABytes, b_lbo, 1024);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16_ss(d, da + a_step * kk, db + b_step * kk, idesc, (kb | kk) != 0);
          mma_commit(ctl.bar(B_EMPTY + st));
        }
        if (ok) mma_commit(ctl.bar(B_ACC_FULL + acc));
      }
      mma_commit(ctl.bar(B_DONE));
      ctl.drain(B_DONE, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int r = (warp & 3) * 32 + lane;  // tile row = TMEM lane
    const uint32_t lane_base = uint32_t(32 * (warp & 3)) << 16;
    uint32_t lt = 0;
    for (int t = blockIdx.x; t < n_tiles_total; t += gridDim.x, ++lt) {
      int m0, n0;
      s.tile(t, m0, n0);
      const uint32_t acc = lt & 1;
      if (!ctl.wait_warp(B_ACC_FULL + acc, (lt >> 1) & 1)) break;
      tc_fence_after();
      // hands the accumulator back to the MMA warp once the epilogue has read it
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ctl.bar(B_ACC_EMPTY + acc));
      };
      epi(tmem + lane_base + acc * kBN, r, m0, n0, release);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// 32 accumulator columns of this thread's row as floats.
__device__ __forceinline__ void acc_chunk(uint32_t ta, int c, float (&v)[32]) {
  uint32_t x[32];
  tmem_ld32(ta + 32 * c, x);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(x[j]);
}

// v[j] = (j == idx) ? v[j] + add : v[j], as an opaque select: written as a
// plain ?: chain over j the compiler turns it into an indexed local-memory copy.
__device__ __forceinline__ void add_at(float (&v)[32], int idx, float add) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    asm("{\n\t.reg .pred p;\n\tsetp.eq.s32 p, %1, %2;\n\t@p add.f32 %0, %0, %3;\n\t}"
        : "+f"(v[j])
        : "r"(j), "r"(idx), "f"(add));
}
__device__ __forceinline__ float pick_at(const float (&v)[32], int idx, float fallback) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    asm("{\n\t.reg .pred p;\n\tsetp.eq.s32 p, %2, %3;\n\tselp.f32 %0, %1, %0, p;\n\t}"
        : "+f"(fallback)
        : "f"(v[j]), "r"(j), "r"(idx));
  return fallback;
}

// Forward epilogue (logits tile of 128 actions x 256 vocabulary entries): the
// row maximum and sum of exponentials of the tile and the label's logit.
struct LseEpi {
  int32_t E, V;
  const int32_t *labels;
  float2 *partial;     // [n_tiles][E]
  float *label_logit;  // [E]
  template <class Release>
  __device__ __forceinline__ void operator()(uint32_t ta, int r, int m0, int n0, Release &release) const {
    const int e = m0 + r, nt = n0 / kBN;
    const bool row_ok = e < E;
    const int yc = (row_ok ? __ldg(labels + e) : -1) - n0;  // label column within the tile
    float m = -INFINITY, sum = 0.f, lab = 0.f;
    const bool tail = n0 + kBN > V;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      float v[32];
      acc_chunk(ta, c, v);
      if (tail) {
        const int lim = V - (n0 + 32 * c);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = j < lim ? v[j] : -INFINITY;
      }
      if ((yc >> 5) == c) lab = pick_at(v, yc & 31, lab);
      float cm = v[0];
#pragma unroll
      for (int j = 1; j < 32; ++j) cm = fmaxf(cm, v[j]);
      if (cm > m) {
        sum *= ex2((m - cm) * kL2e);
        m = cm;
      }
      const float nm = -m * kL2e;
      float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 32; ++j) p[j & 3] += ex2(fmaf(v[j], kL2e, nm));
      sum += (p[0] + p[1]) + (p[2] + p[3]);
    }
    release();
    if (row_ok) {
      partial[size_t(nt) * E + e] = make_float2(m, sum);
      if (yc >= 0 && yc < kBN) label_logit[e] = lab;
    }
  }
};

// Backward epilogue, same tiles: dlogits = g * (onehot(label) - exp(logit - lse)), bf16.
struct DlogitsEpi {
  int32_t E, V;
  const int32_t *labels;
  const float *lse, *grad;
  __nv_bfloat16 *dl;  // [E][V]
  int32_t *d_status;
  template <class Release>
  __device__ __forceinline__ void operator()(uint32_t ta, int r, int m0, int n0, Release &release) const {
    const int e = m0 + r;
    const bool row_ok = e < E;
    int y = -1;
    float nl = 0.f, g = 0.f;
    if (row_ok) {
      y = __ldg(labels + e);
      nl = -__ldg(lse + e) * kL2e;
      g = __ldg(grad + e);
      if (n0 == 0 && (y < 0 || y >= V) && d_status) atomicOr(d_status, SP_DEV_INDEX_RANGE);
    }
    const int yc = y - n0;
    __nv_bfloat16 *row = dl + size_t(e) * V + n0;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      float v[32];
      acc_chunk(ta, c, v);
      if (c == kBN / 32 - 1) release();
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = -g * ex2(fmaf(v[j], kL2e, nl));
      if ((yc >> 5) == c) add_at(v, yc & 31, g);
      if (row_ok) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (n0 + 32 * c + 8 * q < V) {
            uint4 u;
            u.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
            u.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
            u.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
            u.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
            *reinterpret_cast<uint4 *>(row + 32 * c + 8 * q) = u;
          }
        }
      }
    }
  }
};

// Plain fp32 store of the tile into out[M][N] (row stride N).
struct StoreEpi {
  int32_t M, N;
  float *out;
  template <class Release>
  __device__ __forceinline__ void operator()(uint32_t ta, int r, int m0, int n0, Release &release) const {
    const int m = m0 + r;
    float *row = out + size_t(m) * N + n0;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      float v[32];
      acc_chunk(ta, c, v);
      if (c == kBN / 32 - 1) release();
      if (m < M) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (n0 + 32 * c + 4 * q < N)
            *reinterpret_cast<float4 *>(row + 32 * c + 4 * q) =
                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    }
  }
};

// One warp per action: merge the per-tile (max, sum) pairs into lse, then
// logprob = label logit - lse.  A label outside [0, V) sets
// SP_DEV_INDEX_RANGE and yields NaN for that action.
__global__ void __launch_bounds__(256) lmh_combine_kernel(const float2 *__restrict__ partial, int32_t n_tiles,
                                                          int32_t E, int32_t V, const int32_t *__restrict__ labels,
                                                          const float *__restrict__ label_logit, float *logprob,
                                                          float *lse, int32_t *d_status) {
  const int lane = threadIdx.x & 31;
  for (int e = (blockIdx.x * 256 + threadIdx.x) / 32; e < E; e += gridDim.x * 8) {
    float m = -INFINITY, sum = 0.f;
    for (int nt = lane; nt < n_tiles; nt += 32) {
      const float2 p = partial[size_t(nt) * E + e];
      if (p.x > m) {
        sum = sum * ex2((m - p.x) * kL2e) + p.y;
        m = p.x;
      } else {
        sum += p.y * ex2((p.x - m) * kL2e);
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m, off), os = __shfl_xor_sync(0xffffffffu, sum, off);
      const float nm = fmaxf(m, om);
      sum = (nm == -INFINITY) ? 0.f : sum * ex2((m - nm) * kL2e) + os * ex2((om - nm) * kL2e);
      m = nm;
    }
    if (lane == 0) {
      const float l = m + log2f(sum) * kLn2;
      const int y = labels[e];
      const bool ok = y >= 0 && y < V;
      if (!ok && d_status) atomicOr(d_status, SP_DEV_INDEX_RANGE);
      lse[e] = l;
      logprob[e] = ok ? label_logit[e] - l : __int_as_float(0x7fc00000);
    }
  }
}

template <bool A_MN, bool B_MN, class Epi>
int launch_gemm(const CUtensorMap &ta, const CUtensorMap &tb, const GemmShape &s, const Epi &epi, int32_t *d_status,
                int sms, cudaStream_t st) {
  auto kern = gemm_kernel<A_MN, B_MN, Epi>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM_ALLOC) != cudaSuccess)
    return SP_ERR_CUDA;
  const int tiles = s.m_tiles * s.n_tiles;
  kern<<<std::min(tiles, sms), kThreads, SM_ALLOC, st>>>(ta, tb, s, epi, d_status);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

GemmShape gemm_shape(int32_t M, int32_t N, int32_t K, int32_t m_fast) {
  return {M, N, K, (M + kBM - 1) / kBM, (N + kBN - 1) / kBN, (K + kBK - 1) / kBK, m_fast};
}

int sm_count(int *sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SP_ERR_CUDA;
  return SP_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t lmh_workspace(int32_t E, int32_t V) {
  const size_t nt = (size_t(V) + kBN - 1) / kBN;
  return align256(nt * size_t(E) * sizeof(float2)) + align256(size_t(E) * sizeof(float));
}

int lmh_fwd(const void *hidden_sel, int32_t E, int32_t Hd, const void *weight, int32_t V, const int32_t *labels,
            float *logprob, float *lse, void *workspace, int32_t *d_status, void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if (int rc = sm_count(&sms)) return rc;
  // logits[E][V]: A = hidden_sel (K-major), B = weight (K-major), vocabulary blocks outer
  const GemmShape s = gemm_shape(E, V, Hd, 1);
  float2 *partial = static_cast<float2 *>(workspace);
  float *label_logit =
      reinterpret_cast<float *>(static_cast<char *>(workspace) + align256(size_t(s.n_tiles) * E * sizeof(float2)));
  CUtensorMap th, tw;
  int rc = encode_bf16_2d(&th, hidden_sel, Hd, E, kBK, kBM);
  if (!rc) rc = encode_bf16_2d(&tw, weight, Hd, V, kBK, kBN);
  if (!rc) rc = launch_gemm<false, false>(th, tw, s, LseEpi{E, V, labels, partial, label_logit}, d_status, sms, st);
  if (rc) return rc;
  const int cgrid = std::max(1, std::min((E + 7) / 8, sms * 8));
  lmh_combine_kernel<<<cgrid, 256, 0, st>>>(partial, s.n_tiles, E, V, labels, label_logit, logprob, lse, d_status);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

size_t lmh_bwd_workspace(int32_t E, int32_t V) { return align256(size_t(E) * size_t(V) * 2); }

int lmh_bwd(const void *hidden_sel, int32_t E, int32_t Hd, const void *weight, int32_t V, const int32_t *labels,
            const float *lse, const float *grad_logprob, float *d_hidden_sel, float *d_weight, void *workspace,
            int32_t *d_status, void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if (int rc = sm_count(&sms)) return rc;
  __nv_bfloat16 *dl = static_cast<__nv_bfloat16 *>(workspace);
  CUtensorMap th, tw;
  // 1. dlogits[E][V] = g (onehot - softmax), recomputing the logits
  int rc = encode_bf16_2d(&th, hidden_sel, Hd, E, kBK, kBM);
  if (!rc) rc = encode_bf16_2d(&tw, weight, Hd, V, kBK, kBN);
  if (!rc)
    rc = launch_gemm<false, false>(th, tw, gemm_shape(E, V, Hd, 1),
                                   DlogitsEpi{E, V, labels, lse, grad_logprob, dl, d_status}, d_status, sms, st);
  if (rc) return rc;
  // 2. d_hidden_sel[E][Hd] = dlogits[E][V] weight[V][Hd]: A K-major, B MN-major (K = V)
  if (d_hidden_sel) {
    CUtensorMap ta, tb;
    rc = encode_bf16_2d(&ta, dl, V, E, kBK, kBM);
    if (!rc) rc = encode_bf16_2d(&tb, weight, Hd, V, 64, kBK);
    if (!rc) rc = launch_gemm<false, true>(ta, tb, gemm_shape(E, Hd, V, 1), StoreEpi{E, Hd, d_hidden_sel}, d_status,
                                           sms, st);
    if (rc) return rc;
  }
  // 3. d_weight[V][Hd] = dlogits^T[V][E] hidden_sel[E][Hd]: both MN-major (K = E),
  //    the Hd blocks of one vocabulary block side by side so they share its dlogits
  if (d_weight) {
    CUtensorMap ta, tb;
    rc = encode_bf16_2d(&ta, dl, V, E, 64, kBK);
    if (!rc) rc = encode_bf16_2d(&tb, hidden_sel, Hd, E, 64, kBK);
    if (!rc) rc = launch_gemm<true, true>(ta, tb, gemm_shape(V, Hd, E, 0), StoreEpi{V, Hd, d_weight}, d_status,
                                          sms, st);
    if (rc) return rc;
  }
  return SP_OK;
}

}  // namespace spc
