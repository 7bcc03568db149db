// Vocabulary head over the sampled-edge states: per-action log-probability of
// the sampled token ("[ENHANCEMENT] Shared-prefix training with context
// parallelism for exact agent trajectories", issue #7386, "Describe the
// solution you'd like", fifth bullet: only sampled-edge source states are
// projected, one loss owner per sampled action; "TreePackedSeqParams" draft,
// PR #7387, "Summary": edge-source selection before the vocabulary projection).
//
//   logits[e][v] = <h[e], W[v]>    (h: [E][Hd], W: [V][Hd], bf16; fp32 accumulation)
//   lse[e]       = log sum_v exp(logits[e][v])
//   logprob[e]   = logits[e][labels[e]] - lse[e]
//
// lmh_fwd_kernel: persistent tcgen05 GEMM over 128-action x 256-vocabulary
// tiles, vocabulary-block-major so that CTAs running side by side read the
// same W block (from L2) while h stays L2-resident.  A 4-stage TMA ring feeds
// 128x256x16 MMAs into one of two 256-column TMEM accumulators; the epilogue
// warpgroup (thread = action row = TMEM lane) reduces the other accumulator to
// the tile's row maximum and sum of exponentials and picks out the label's
// logit, so the [E][V] logits never reach memory.  lmh_combine_kernel merges
// the per-tile partials into lse and logprob.
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

struct LmhShape {
  int32_t E, V, Hd;
  int32_t m_tiles, n_tiles, k_blocks;
};

__global__ void __launch_bounds__(kThreads, 1)
    lmh_fwd_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w, LmhShape s,
                   const int32_t *__restrict__ labels, float2 *__restrict__ partial, float *__restrict__ label_logit,
                   int32_t *d_status) {
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
      prefetch_tmap(&tm_h);
      prefetch_tmap(&tm_w);
      uint32_t it = 0;  // stage fills issued
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles_total; t += gridDim.x) {
        const int m0 = (t % s.m_tiles) * kBM, n0 = (t / s.m_tiles) * kBN;
        for (int kb = 0; kb < s.k_blocks; ++kb, ++it) {
          const uint32_t st = it % kStages, ph = (it / kStages) & 1;
          if (!(ok = ctl.wait(B_EMPTY + st, ph ^ 1))) break;
          const uint32_t dst = sbase + st * kStage;
          mbar_arrive_expect_tx(ctl.bar(B_FULL + st), kStage);
          tma_load_2d(dst, &tm_h, ctl.bar(B_FULL + st), kb * kBK, m0);
          tma_load_2d(dst + kABytes, &tm_w, ctl.bar(B_FULL + st), kb * kBK, n0);
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
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, 0, 0);
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
          const uint64_t da = smem_desc_sw128(sbase + st * kStage, 16, 1024);
          const uint64_t db = smem_desc_sw128(sbase + st * kStage + kABytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) mma_bf16_ss(d, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) != 0);
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
      const int mt = t % s.m_tiles, nt = t / s.m_tiles;
      const int e = mt * kBM + r, n0 = nt * kBN;
      const bool row_ok = e < s.E;
      const int yc = (row_ok ? __ldg(labels + e) : -1) - n0;  // label column within the tile
      const uint32_t acc = lt & 1;
      if (!ctl.wait_warp(B_ACC_FULL + acc, (lt >> 1) & 1)) break;
      tc_fence_after();
      const uint32_t ta = tmem + lane_base + acc * kBN;
      float m = -INFINITY, sum = 0.f, lab = 0.f;
      const bool tail = n0 + kBN > s.V;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t x[32];
        tmem_ld32(ta + 32 * c, x);
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(x[j]);
        if (tail) {
          const int lim = s.V - (n0 + 32 * c);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = j < lim ? v[j] : -INFINITY;
        }
        if ((yc >> 5) == c) {
          // an opaque select: written as a plain ?: the compiler turns the
          // chain into an indexed load from a local-memory copy of v
#pragma unroll
          for (int j = 0; j < 32; ++j)
            asm("{\n\t.reg .pred p;\n\tsetp.eq.s32 p, %2, %3;\n\tselp.f32 %0, %1, %0, p;\n\t}"
                : "+f"(lab)
                : "f"(v[j]), "r"(j), "r"(yc & 31));
        }
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
      // accumulator drained: hand it back to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ctl.bar(B_ACC_EMPTY + acc));
      if (row_ok) {
        partial[size_t(nt) * s.E + e] = make_float2(m, sum);
        if (yc >= 0 && yc < kBN) label_logit[e] = lab;
      }
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

}  // namespace

size_t lmh_workspace(int32_t E, int32_t V) {
  const size_t nt = (size_t(V) + kBN - 1) / kBN;
  const auto a = [](size_t x) { return (x + 255) & ~size_t(255); };
  return a(nt * size_t(E) * sizeof(float2)) + a(size_t(E) * sizeof(float));
}

int lmh_fwd(const void *hidden_sel, int32_t E, int32_t Hd, const void *weight, int32_t V, const int32_t *labels,
            float *logprob, float *lse, void *workspace, int32_t *d_status, void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SP_ERR_CUDA;
  LmhShape s{E, V, Hd, (E + kBM - 1) / kBM, (V + kBN - 1) / kBN, (Hd + kBK - 1) / kBK};
  const auto a = [](size_t x) { return (x + 255) & ~size_t(255); };
  float2 *partial = static_cast<float2 *>(workspace);
  float *label_logit =
      reinterpret_cast<float *>(static_cast<char *>(workspace) + a(size_t(s.n_tiles) * E * sizeof(float2)));

  CUtensorMap th, tw;
  int rc = encode_bf16_2d(&th, hidden_sel, Hd, E, kBK, kBM);
  if (!rc) rc = encode_bf16_2d(&tw, weight, Hd, V, kBK, kBN);
  if (rc) return rc;
  if (cudaFuncSetAttribute(lmh_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SM_ALLOC) != cudaSuccess)
    return SP_ERR_CUDA;
  const int tiles = s.m_tiles * s.n_tiles;
  const int grid = std::min(tiles, sms);
  lmh_fwd_kernel<<<grid, kThreads, SM_ALLOC, st>>>(th, tw, s, labels, partial, label_logit, d_status);
  if (cudaGetLastError() != cudaSuccess) return SP_ERR_CUDA;
  const int cgrid = std::max(1, std::min((E + 7) / 8, sms * 8));
  lmh_combine_kernel<<<cgrid, 256, 0, st>>>(partial, s.n_tiles, E, V, labels, label_logit, logprob, lse, d_status);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

}  // namespace spc
