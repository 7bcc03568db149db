// Sampled-edge source selection: out[e] = hidden[idx[e]] (issue #7386,
// "Describe the solution you'd like", fifth bullet, and PR #7387 "Summary",
// fourth bullet: only edge-source hidden states go to the vocabulary head).
//
// A pure row copy, bound by HBM bandwidth: one warp per output row, 16-byte
// vector loads and stores, several independent loads in flight per lane.
// The grid is a multiple of the SM count and strides over the rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

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

// ---------------------------------------------------------------------------
// Backward of the gather: grad_hidden[t] = sum of grad_out[e] over the actions
// e whose source is t (zero for tokens that are no action's source).  Several
// actions can share a source token (a branch point), so the rows are summed in
// ascending e -- the same order on every run.  Steps (workspace: cnt, fill,
// off[T+1], list[E]): count sources per token, exclusive prefix sum, bucket the
// actions per token (slot order from atomics is arbitrary), then one warp per
// token orders its bucket by e and sums in that order in fp32.
namespace spc {
namespace {

__global__ void __launch_bounds__(kThreads) gb_zero_kernel(int32_t *p, long n) {
  for (long i = long(blockIdx.x) * kThreads + threadIdx.x; i < n; i += long(gridDim.x) * kThreads) p[i] = 0;
}

__global__ void __launch_bounds__(kThreads) gb_count_kernel(const int32_t *__restrict__ idx, int32_t E, int32_t T,
                                                            int32_t *cnt, int32_t *d_status) {
  for (int e = blockIdx.x * kThreads + threadIdx.x; e < E; e += gridDim.x * kThreads) {
    const int32_t t = __ldg(idx + e);
    if (t < 0 || t >= T) {
      if (d_status) atomicOr(d_status, SP_DEV_INDEX_RANGE);
      continue;
    }
    atomicAdd(cnt + t, 1);
  }
}

// off[0] = 0, off[t + 1] = off[t] + cnt[t]; one CTA, 1024-token chunks.
__global__ void __launch_bounds__(1024) gb_scan_kernel(const int32_t *__restrict__ cnt, int32_t T, int32_t *off) {
  __shared__ int32_t warp_sum[32];
  __shared__ int32_t carry;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    carry = 0;
    off[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < T; base += 1024) {
    const int t = base + threadIdx.x;
    const int32_t x = t < T ? cnt[t] : 0;
    int32_t inc = x;  // inclusive scan within the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, inc, d);
      if (lane >= d) inc += y;
    }
    if (lane == 31) warp_sum[w] = inc;
    __syncthreads();
    if (w == 0) {
      int32_t s = warp_sum[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, s, d);
        if (lane >= d) s += y;
      }
      warp_sum[lane] = s;  // inclusive over warps
    }
    __syncthreads();
    const int32_t before = carry + (w > 0 ? warp_sum[w - 1] : 0);
    if (t < T) off[t + 1] = before + inc;
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_sum[31];
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads) gb_fill_kernel(const int32_t *__restrict__ idx, int32_t E, int32_t T,
                                                           const int32_t *__restrict__ off, int32_t *fill,
                                                           int32_t *list) {
  for (int e = blockIdx.x * kThreads + threadIdx.x; e < E; e += gridDim.x * kThreads) {
    const int32_t t = __ldg(idx + e);
    if (t < 0 || t >= T) continue;
    list[off[t] + atomicAdd(fill + t, 1)] = e;
  }
}

template <typename Tv>
__device__ __forceinline__ void add8(float (&a)[8], const Tv *p);
template <>
__device__ __forceinline__ void add8<float>(float (&a)[8], const float *p) {
  const float4 x = *reinterpret_cast<const float4 *>(p), y = *reinterpret_cast<const float4 *>(p + 4);
  a[0] += x.x, a[1] += x.y, a[2] += x.z, a[3] += x.w, a[4] += y.x, a[5] += y.y, a[6] += y.z, a[7] += y.w;
}
template <>
__device__ __forceinline__ void add8<__nv_bfloat16>(float (&a)[8], const __nv_bfloat16 *p) {
  const uint4 u = *reinterpret_cast<const uint4 *>(p);
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    a[2 * i] += f.x, a[2 * i + 1] += f.y;
  }
}
__device__ __forceinline__ void store8(float *p, const float (&a)[8]) {
  *reinterpret_cast<float4 *>(p) = make_float4(a[0], a[1], a[2], a[3]);
  *reinterpret_cast<float4 *>(p + 4) = make_float4(a[4], a[5], a[6], a[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float (&a)[8]) {
  uint4 u;
  uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&h);
  }
  *reinterpret_cast<uint4 *>(p) = u;
}

// One warp per token: order the bucket by action index, then sum its rows.
template <typename Tv>
__global__ void __launch_bounds__(kThreads) gb_reduce_kernel(const Tv *__restrict__ grad_out, int32_t hidden_dim,
                                                             int32_t T, const int32_t *__restrict__ off,
                                                             int32_t *list, Tv *__restrict__ grad_hidden) {
  const int lane = threadIdx.x & 31;
  for (int t = blockIdx.x * kWarps + (threadIdx.x >> 5); t < T; t += gridDim.x * kWarps) {
    const int32_t b = off[t], n = off[t + 1] - b;
    int32_t *bucket = list + b;
    if (n > 1 && lane == 0) {  // insertion sort: buckets hold the few actions sharing one token
      for (int i = 1; i < n; ++i) {
        const int32_t x = bucket[i];
        int j = i - 1;
        while (j >= 0 && bucket[j] > x) {
          bucket[j + 1] = bucket[j];
          --j;
        }
        bucket[j + 1] = x;
      }
    }
    __syncwarp();
    Tv *dst = grad_hidden + size_t(t) * hidden_dim;
    for (int c = lane * 8; c < hidden_dim; c += 256) {
      float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int i = 0; i < n; ++i) add8(a, grad_out + size_t(bucket[i]) * hidden_dim + c);
      store8(dst + c, a);
    }
  }
}

}  // namespace

size_t edge_gather_bwd_workspace(int32_t T, int32_t E) {
  const auto a = [](size_t x) { return (x + 255) & ~size_t(255); };
  return a(size_t(T) * 4) * 2 + a(size_t(T + 1) * 4) + a(size_t(E) * 4);
}

int edge_gather_bwd(int32_t elem_bytes, const void *grad_out, int32_t E, int32_t hidden_dim, const int32_t *idx,
                    int32_t T, void *grad_hidden, void *workspace, int32_t *d_status, void *stream) {
  if (hidden_dim % 8) return SP_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SP_ERR_CUDA;
  const auto a = [](size_t x) { return (x + 255) & ~size_t(255); };
  char *w = static_cast<char *>(workspace);
  int32_t *cnt = reinterpret_cast<int32_t *>(w);
  int32_t *fill = reinterpret_cast<int32_t *>(w + a(size_t(T) * 4));
  int32_t *off = reinterpret_cast<int32_t *>(w + 2 * a(size_t(T) * 4));
  int32_t *list = reinterpret_cast<int32_t *>(w + 2 * a(size_t(T) * 4) + a(size_t(T + 1) * 4));
  const int g_small = std::max(1, std::min(sms * 4, int((2 * long(T) + kThreads - 1) / kThreads)));
  // cnt and fill are adjacent 256-byte-aligned arrays: zero both in one pass
  gb_zero_kernel<<<g_small, kThreads, 0, st>>>(cnt, long(a(size_t(T) * 4) / 4) * 2);
  if (E > 0) {
    const int ge = std::max(1, std::min(sms * 4, (E + kThreads - 1) / kThreads));
    gb_count_kernel<<<ge, kThreads, 0, st>>>(idx, E, T, cnt, d_status);
    gb_scan_kernel<<<1, 1024, 0, st>>>(cnt, T, off);
    gb_fill_kernel<<<ge, kThreads, 0, st>>>(idx, E, T, off, fill, list);
  } else {
    gb_zero_kernel<<<g_small, kThreads, 0, st>>>(off, long(T) + 1);
  }
  const int gr = std::max(1, std::min(sms * 8, (T + kWarps - 1) / kWarps));
  if (elem_bytes == 2)
    gb_reduce_kernel<__nv_bfloat16><<<gr, kThreads, 0, st>>>(static_cast<const __nv_bfloat16 *>(grad_out),
                                                             hidden_dim, T, off, list,
                                                             static_cast<__nv_bfloat16 *>(grad_hidden));
  else
    gb_reduce_kernel<float><<<gr, kThreads, 0, st>>>(static_cast<const float *>(grad_out), hidden_dim, T, off, list,
                                                     static_cast<float *>(grad_hidden));
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

}  // namespace spc
