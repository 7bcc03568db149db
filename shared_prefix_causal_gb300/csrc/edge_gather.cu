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

// off[0] = 0, off[t + 1] = off[t] + cnt[t]; one CTA over chunks of 8192
// tokens: thread i scans tokens [8i, 8i+8) of the chunk (two 16-byte loads,
// coalesced across the warp), one block-wide scan of the thread totals, and a
// carry from chunk to chunk.
__global__ void __launch_bounds__(1024) gb_scan_kernel(const int32_t *__restrict__ cnt, int32_t T, int32_t *off) {
  __shared__ int32_t warp_sum[32];
  __shared__ int32_t carry;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    carry = 0;
    off[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < T; base += 8192) {
    const int t0 = base + 8 * int(threadIdx.x);
    int32_t x[8];
    if (t0 + 8 <= T) {
      const int4 a = *reinterpret_cast<const int4 *>(cnt + t0), b = *reinterpret_cast<const int4 *>(cnt + t0 + 4);
      x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = t0 + k < T ? cnt[t0 + k] : 0;
    }
#pragma unroll
    for (int k = 1; k < 8; ++k) x[k] += x[k - 1];  // inclusive within the thread
    int32_t inc = x[7];                           // inclusive over the warp's threads
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, inc, d);
      if (lane >= d) inc += y;
    }
    if (lane == 31) warp_sum[w] = inc;
    __syncthreads();
    if (w == 0) {
      int32_t v = warp_sum[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += y;
      }
      warp_sum[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    const int32_t before = carry + (w > 0 ? warp_sum[w - 1] : 0) + inc - x[7];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (t0 + k < T) off[t0 + k + 1] = before + x[k];
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

// 16 bytes of a row: 4 fp32 or 8 bf16 values, accumulated in fp32.
template <typename Tv>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void add(float (&a)[N], const float *p) {
    const float4 x = *reinterpret_cast<const float4 *>(p);
    a[0] += x.x, a[1] += x.y, a[2] += x.z, a[3] += x.w;
  }
  static __device__ __forceinline__ void store(float *p, const float (&a)[N]) {
    *reinterpret_cast<float4 *>(p) = make_float4(a[0], a[1], a[2], a[3]);
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void add(float (&a)[N], const __nv_bfloat16 *p) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      a[2 * i] += f.x, a[2 * i + 1] += f.y;
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float (&a)[N]) {
    uint4 u;
    uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(p) = u;
  }
};

// One warp per token: order the bucket by action index, then sum its rows.
// Each lane owns 16 consecutive bytes of every 512-byte stretch of the row,
// so a warp's loads and stores cover whole sectors.
template <typename Tv>
__global__ void __launch_bounds__(kThreads) gb_reduce_kernel(const Tv *__restrict__ grad_out, int32_t hidden_dim,
                                                             int32_t T, const int32_t *__restrict__ off,
                                                             int32_t *list, Tv *__restrict__ grad_hidden) {
  using V16 = Vec16<Tv>;
  constexpr int kN = V16::N;
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
    for (int c = lane * kN; c < hidden_dim; c += 32 * kN) {
      float a[kN];
#pragma unroll
      for (int i = 0; i < kN; ++i) a[i] = 0.f;
      for (int i = 0; i < n; ++i) V16::add(a, grad_out + size_t(bucket[i]) * hidden_dim + c);
      V16::store(dst + c, a);
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
