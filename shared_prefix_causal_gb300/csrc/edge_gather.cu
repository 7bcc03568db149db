// Sampled-edge source selection: out[e] = hidden[idx[e]] (issue #7386,
// "Describe the solution you'd like", fifth bullet, and PR #7387 "Summary",
// fourth bullet: only edge-source hidden states go to the vocabulary head).
//
// A pure row copy, bound by HBM bandwidth: one warp per output row, 16-byte
// vector loads and stores, several independent loads in flight per lane.
// The grid is a multiple of the SM count and strides over the rows.
#include <cuda_runtime.h>

#include "internal.h"

namespace spc {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) edge_gather_kernel(const int4 *__restrict__ hidden, int32_t T,
                                                               int32_t row_vec, const int32_t *__restrict__ idx,
                                                               int32_t E, int4 *__restrict__ out,
                                                               int32_t *d_status) {
  const int lane = threadIdx.x & 31;
  for (int e = blockIdx.x * kWarps + (threadIdx.x >> 5); e < E; e += gridDim.x * kWarps) {
    const int32_t src = __ldg(idx + e);
    int4 *dst = out + size_t(e) * row_vec;
    if (src < 0 || src >= T) {
      for (int c = lane; c < row_vec; c += 32) dst[c] = make_int4(0, 0, 0, 0);
      if (lane == 0 && d_status) atomicOr(d_status, SP_DEV_INDEX_RANGE);
      continue;
    }
    const int4 *row = hidden + size_t(src) * row_vec;
    int c = lane;
    for (; c + 32 * (kUnroll - 1) < row_vec; c += 32 * kUnroll) {
      int4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(row + c + 32 * u);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) __stcs(dst + c + 32 * u, v[u]);
    }
    for (; c < row_vec; c += 32) __stcs(dst + c, __ldcs(row + c));
  }
}

}  // namespace

int edge_gather(int32_t elem_bytes, const void *hidden, int32_t T, int32_t hidden_dim, const int32_t *idx,
                int32_t E, void *out, int32_t *d_status, void *stream) {
  const size_t row_bytes = size_t(hidden_dim) * elem_bytes;
  if (row_bytes % 16) return SP_ERR_UNSUPPORTED;
  if (E == 0) return SP_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SP_ERR_CUDA;
  const int want = (E + kWarps - 1) / kWarps;
  const int grid = want < sms * 8 ? want : sms * 8;
  edge_gather_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const int4 *>(hidden), T, int32_t(row_bytes / 16), idx, E, static_cast<int4 *>(out), d_status);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

}  // namespace spc
