// The default backward's two companion kernels on sm_103a, memory-bound
// elementwise passes around its main kernel:
//   bwd_pre     Delta = rowsum(dO * O) per (token, query head), the softmax
//               backward's per-row term (FlashAttention-style recomputation),
//               and zeroing the fp32 dQ workspace the main kernel adds into;
//   dq_convert  dQ = bf16(scale * workspace).
// The backward sums every branch's contribution into the prefix the branches
// share (#7914, "feat(hybrid): add opt-in shared-prefix attention and Mamba
// execution", introduction); these passes touch each row once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace spc {
namespace {

using namespace ptx;

// Delta = rowsum(dO * O) per (token, query head) in fp32, and zero the fp32
// dQ workspace (when there is one).  A row of D values is read by D / 8 lanes
// with 16-byte loads, so a warp takes 256 / D rows at once and every lane loads.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16 *__restrict__ o,
                                                      const __nv_bfloat16 *__restrict__ d_o,
                                                      float *__restrict__ delta, float *__restrict__ dqacc, int T,
                                                      int Hq) {
  constexpr int kLanes = D / 8;            // lanes per row
  constexpr int kRowsPerWarp = 32 / kLanes;
  const int lane = threadIdx.x & 31, sub = lane / kLanes, part = lane % kLanes;
  const long rows = long(T) * Hq;
  const long warp0 = (long(blockIdx.x) * 256 + threadIdx.x) / 32, warps = long(gridDim.x) * 8;
  for (long row0 = warp0 * kRowsPerWarp; row0 < rows; row0 += warps * kRowsPerWarp) {
    const long row = row0 + sub;
    const bool live = row < rows;
    float acc = 0.f;
    if (live) {
      const uint4 a = *reinterpret_cast<const uint4 *>(o + row * D + part * 8);
      const uint4 b = *reinterpret_cast<const uint4 *>(d_o + row * D + part * 8);
      const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
      const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&b);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(pa[i]), y = __bfloat1622float2(pb[i]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
      if (dqacc) {
        float4 *z = reinterpret_cast<float4 *>(dqacc + row * D) + 2 * part;
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int off = kLanes / 2; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (live && part == 0) delta[size_t(row % Hq) * T + row / Hq] = acc;
  }
}

// dq = bf16(scale * dqacc), 8 elements per thread per step.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float *__restrict__ dqacc,
                                                         __nv_bfloat16 *__restrict__ dq, float scale, long n8) {
  for (long i = long(blockIdx.x) * 256 + threadIdx.x; i < n8; i += long(gridDim.x) * 256) {
    const float4 a = reinterpret_cast<const float4 *>(dqacc)[2 * i];
    const float4 b = reinterpret_cast<const float4 *>(dqacc)[2 * i + 1];
    uint4 w;
    w.x = pack_bf16(a.x * scale, a.y * scale);
    w.y = pack_bf16(a.z * scale, a.w * scale);
    w.z = pack_bf16(b.x * scale, b.y * scale);
    w.w = pack_bf16(b.z * scale, b.w * scale);
    reinterpret_cast<uint4 *>(dq)[i] = w;
  }
}

}  // namespace

int bwd_pre(const AttnShape &s, const void *o, const void *d_o, float *delta, float *dqacc, int sms,
            void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long rows = long(s.T) * s.Hq;
  const int grid = int(std::min<long>((rows + 7) / 8, long(sms) * 16));
  const auto *po = static_cast<const __nv_bfloat16 *>(o);
  const auto *pdo = static_cast<const __nv_bfloat16 *>(d_o);
  if (s.D == 128)
    bwd_pre_kernel<128><<<grid, 256, 0, st>>>(po, pdo, delta, dqacc, s.T, s.Hq);
  else if (s.D == 64)
    bwd_pre_kernel<64><<<grid, 256, 0, st>>>(po, pdo, delta, dqacc, s.T, s.Hq);
  else
    return SP_ERR_UNSUPPORTED;
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

int dq_convert(const float *dqacc, void *dq, float scale, long n, int sms, void *stream) {
  const long n8 = n / 8;
  const int grid = int(std::min<long>((n8 + 255) / 256, long(sms) * 16));
  dq_convert_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(dqacc, static_cast<__nv_bfloat16 *>(dq),
                                                                          scale, n8);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

}  // namespace spc
