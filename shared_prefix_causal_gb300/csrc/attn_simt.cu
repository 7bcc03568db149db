// Tree attention on the CUDA cores in fp32 (the fp32-input mode).
//
// Same plan walk as the tensor-core path: a query tile reads the key ranges
// of its ancestors (fully visible) and its own segment up to the tile end
// (causal), as PR #7387 "TreePackedSeqParams", "Summary" has a query segment
// attend over its ancestors.  The backward is split in two
// deterministic kernels: dQ walks the same forward ranges; dK/dV walks, for
// each block of keys, the one contiguous run of queries that can see it (the
// key's segment and its whole subtree, which preorder places right after it),
// so every branch's contribution is summed into the shared prefix (#7914,
// introduction).
//
// Work decomposition: a CTA of 256 threads owns 64 rows (query rows of a
// tile for the forward and dQ, keys of a block for dK/dV) and steps over the
// other side 32 at a time.  Thread t handles row t/4; for 64x32 score blocks
// it computes columns (t%4) + 4m, m < 8; for 64xD accumulators it holds
// columns 16i + 4(t%4) .. +3.  Operands are staged in shared memory as fp32
// with rows padded by 4 floats, which keeps every access conflict-free.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "internal.h"

namespace spc {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 64;
constexpr int kCols = 32;
constexpr int kPStride = kCols + 1;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
  const uint2 u = *reinterpret_cast<const uint2 *>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t *>(&a);
  u.y = *reinterpret_cast<uint32_t *>(&b);
  *reinterpret_cast<uint2 *>(p) = u;
}

__device__ __forceinline__ void flag(int32_t *d_status, int bit) {
  if (d_status) atomicOr(d_status, bit);
}

// Stage `nrows` rows of a [T][H][D] tensor into smem [nrows][D+4] (fp32).
// Row r maps to (token, head) through row_src; rows with token < 0 are zero.
template <typename Tin, int D, typename F>
__device__ __forceinline__ void stage_rows(float *dst, const Tin *src, int nrows, int H, F row_src) {
  constexpr int kV = D / 4;
  for (int idx = threadIdx.x; idx < nrows * kV; idx += kThreads) {
    const int r = idx / kV, c = (idx % kV) * 4;
    int tok, head;
    row_src(r, tok, head);
    float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tok >= 0) val = load4(src + (size_t(tok) * H + head) * D + c);
    store4(dst + r * (D + 4) + c, val);
  }
}

// s[m] = <A[r], B[x + 4m]>, m < 8.
template <int D>
__device__ __forceinline__ void scores(const float *A, const float *B, int r, int x, float s[8]) {
#pragma unroll
  for (int m = 0; m < 8; ++m) s[m] = 0.f;
  const float *a = A + r * (D + 4);
#pragma unroll 4
  for (int d = 0; d < D; d += 4) {
    const float4 av = load4(a + d);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float4 bv = load4(B + (x + 4 * m) * (D + 4) + d);
      s[m] = fmaf(av.x, bv.x, s[m]);
      s[m] = fmaf(av.y, bv.y, s[m]);
      s[m] = fmaf(av.z, bv.z, s[m]);
      s[m] = fmaf(av.w, bv.w, s[m]);
    }
  }
}

// acc[i] += sum_c P[r][c] * V[c][16i + 4x .. +3], c < 32.
template <int D>
__device__ __forceinline__ void accumulate(float4 *acc, const float *P, const float *V, int r, int x) {
#pragma unroll 4
  for (int c = 0; c < kCols; ++c) {
    const float p = P[r * kPStride + c];
    const float *vr = V + c * (D + 4) + 4 * x;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      const float4 v = load4(vr + 16 * i);
      acc[i].x = fmaf(p, v.x, acc[i].x);
      acc[i].y = fmaf(p, v.y, acc[i].y);
      acc[i].z = fmaf(p, v.z, acc[i].z);
      acc[i].w = fmaf(p, v.w, acc[i].w);
    }
  }
}

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

__device__ __forceinline__ bool range_ok(int a, int b, int T) { return 0 <= a && a <= b && b <= T; }

// ----------------------------------------------------------------- forward
template <typename Tin, int D>
__global__ void __launch_bounds__(kThreads) fwd_kernel(PlanDev plan, AttnShape s, const Tin *__restrict__ q,
                                                       const Tin *__restrict__ k, const Tin *__restrict__ v,
                                                       Tin *__restrict__ o, float *__restrict__ lse,
                                                       int32_t *d_status) {
  extern __shared__ float smem[];
  float *Qs = smem;                        // [64][D+4]
  float *Ks = Qs + kRows * (D + 4);        // [32][D+4]
  float *Vs = Ks + kCols * (D + 4);        // [32][D+4]
  float *Ps = Vs + kCols * (D + 4);        // [64][33]

  const int g = blockIdx.x / plan.n_tiles;
  const int *tile = plan.tiles + 5 * (blockIdx.x % plan.n_tiles);
  const int q0 = tile[1], q1 = tile[2], rb = tile[3], rc = tile[4];
  const int G = s.G, T = s.T;
  const int row0 = blockIdx.y * kRows;
  const int rows_tile = (q1 - q0) * G;
  if (!range_ok(q0, q1, T)) {
    if (threadIdx.x == 0) flag(d_status, SP_DEV_BAD_PLAN);
    return;
  }
  if (row0 >= rows_tile) return;

  stage_rows<Tin, D>(Qs, q, kRows, s.Hq, [&](int r, int &tok, int &head) {
    const int rr = row0 + r;
    tok = rr < rows_tile ? q0 + rr / G : -1;
    head = g * G + rr % G;
  });

  const int r = threadIdx.x >> 2, x = threadIdx.x & 3;
  const int rr = row0 + r;
  const bool rvalid = rr < rows_tile;
  const int tok = q0 + rr / G;
  const int head = g * G + rr % G;
  const float sl2 = s.scale * kLog2e;

  float m_run = -INFINITY, l_run = 0.f;
  float4 acc[D / 16];
#pragma unroll
  for (int i = 0; i < D / 16; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);

  for (int ri = 0; ri < rc; ++ri) {
    const int kv0 = plan.ranges[2 * (rb + ri)], kv1 = plan.ranges[2 * (rb + ri) + 1];
    if (!range_ok(kv0, kv1, T)) {
      if (threadIdx.x == 0) flag(d_status, SP_DEV_BAD_PLAN);
      continue;
    }
    const bool causal = ri == rc - 1;
    for (int kb = kv0; kb < kv1; kb += kCols) {
      __syncthreads();
      auto key_src = [&](int c, int &t_, int &h_) {
        t_ = kb + c < kv1 ? kb + c : -1;
        h_ = g;
      };
      stage_rows<Tin, D>(Ks, k, kCols, s.Hkv, key_src);
      stage_rows<Tin, D>(Vs, v, kCols, s.Hkv, key_src);
      __syncthreads();
      float sc[8];
      scores<D>(Qs, Ks, r, x, sc);
      float bmax = -INFINITY;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int j = kb + x + 4 * m;
        const bool ok = j < kv1 && (!causal || j <= tok);
        sc[m] = ok ? sc[m] * sl2 : -INFINITY;
        bmax = fmaxf(bmax, sc[m]);
      }
      bmax = quad_max(bmax);
      const float m_new = fmaxf(m_run, bmax);
      const float alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
      float psum = 0.f;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const float p = sc[m] == -INFINITY ? 0.f : exp2f(sc[m] - m_new);
        Ps[r * kPStride + x + 4 * m] = p;
        psum += p;
      }
      psum = quad_sum(psum);
      if (m_new != -INFINITY) {
        l_run = l_run * alpha + psum;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
          acc[i].x *= alpha;
          acc[i].y *= alpha;
          acc[i].z *= alpha;
          acc[i].w *= alpha;
        }
        m_run = m_new;
      }
      __syncthreads();
      accumulate<D>(acc, Ps, Vs, r, x);
    }
  }
  if (rvalid) {
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    Tin *orow = o + (size_t(tok) * s.Hq + head) * D + 4 * x;
#pragma unroll
    for (int i = 0; i < D / 16; ++i)
      store4(orow + 16 * i, make_float4(acc[i].x * inv, acc[i].y * inv, acc[i].z * inv, acc[i].w * inv));
    if (x == 0) lse[size_t(head) * T + tok] = (m_run + log2f(l_run)) * kLn2;
  }
}

// ------------------------------------------------- backward: Delta = rowsum(dO*O)
template <typename Tin, int D>
__global__ void __launch_bounds__(kThreads) delta_kernel(AttnShape s, const Tin *__restrict__ o,
                                                         const Tin *__restrict__ d_o, float *__restrict__ delta) {
  const int lane = threadIdx.x & 31;
  const long rows = long(s.T) * s.Hq;
  for (long row = (long(blockIdx.x) * kThreads + threadIdx.x) / 32; row < rows;
       row += long(gridDim.x) * (kThreads / 32)) {
    float acc = 0.f;
    for (int c = lane * 4; c < D; c += 128) {
      const float4 a = load4(o + row * D + c), b = load4(d_o + row * D + c);
      acc += a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      const int tok = int(row / s.Hq), head = int(row % s.Hq);
      delta[size_t(head) * s.T + tok] = acc;
    }
  }
}

// ----------------------------------------------------------- backward: dQ
template <typename Tin, int D>
__global__ void __launch_bounds__(kThreads) dq_kernel(PlanDev plan, AttnShape s, const Tin *__restrict__ q,
                                                      const Tin *__restrict__ k, const Tin *__restrict__ v,
                                                      const Tin *__restrict__ d_o, const float *__restrict__ lse,
                                                      const float *__restrict__ delta, Tin *__restrict__ dq,
                                                      int32_t *d_status) {
  extern __shared__ float smem[];
  float *Qs = smem;                     // [64][D+4]
  float *dOs = Qs + kRows * (D + 4);    // [64][D+4]
  float *Ks = dOs + kRows * (D + 4);    // [32][D+4]
  float *Vs = Ks + kCols * (D + 4);     // [32][D+4]
  float *Ss = Vs + kCols * (D + 4);     // [64][33]

  const int g = blockIdx.x / plan.n_tiles;
  const int *tile = plan.tiles + 5 * (blockIdx.x % plan.n_tiles);
  const int q0 = tile[1], q1 = tile[2], rb = tile[3], rc = tile[4];
  const int G = s.G, T = s.T;
  const int row0 = blockIdx.y * kRows;
  const int rows_tile = (q1 - q0) * G;
  if (!range_ok(q0, q1, T)) {
    if (threadIdx.x == 0) flag(d_status, SP_DEV_BAD_PLAN);
    return;
  }
  if (row0 >= rows_tile) return;
  auto qrow = [&](int r, int &tok, int &head) {
    const int rr = row0 + r;
    tok = rr < rows_tile ? q0 + rr / G : -1;
    head = g * G + rr % G;
  };
  stage_rows<Tin, D>(Qs, q, kRows, s.Hq, qrow);
  stage_rows<Tin, D>(dOs, d_o, kRows, s.Hq, qrow);

  const int r = threadIdx.x >> 2, x = threadIdx.x & 3;
  const int rr = row0 + r;
  const bool rvalid = rr < rows_tile;
  const int tok = q0 + rr / G;
  const int head = g * G + rr % G;
  const float sl2 = s.scale * kLog2e;
  const float lse2 = rvalid ? lse[size_t(head) * T + tok] * kLog2e : 0.f;
  const float dlt = rvalid ? delta[size_t(head) * T + tok] : 0.f;

  float4 acc[D / 16];
#pragma unroll
  for (int i = 0; i < D / 16; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);

  for (int ri = 0; ri < rc; ++ri) {
    const int kv0 = plan.ranges[2 * (rb + ri)], kv1 = plan.ranges[2 * (rb + ri) + 1];
    if (!range_ok(kv0, kv1, T)) {
      if (threadIdx.x == 0) flag(d_status, SP_DEV_BAD_PLAN);
      continue;
    }
    const bool causal = ri == rc - 1;
    for (int kb = kv0; kb < kv1; kb += kCols) {
      __syncthreads();
      auto key_src = [&](int c, int &t_, int &h_) {
        t_ = kb + c < kv1 ? kb + c : -1;
        h_ = g;
      };
      stage_rows<Tin, D>(Ks, k, kCols, s.Hkv, key_src);
      stage_rows<Tin, D>(Vs, v, kCols, s.Hkv, key_src);
      __syncthreads();
      float sc[8], dp[8];
      scores<D>(Qs, Ks, r, x, sc);
      scores<D>(dOs, Vs, r, x, dp);
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int j = kb + x + 4 * m;
        const bool ok = rvalid && j < kv1 && (!causal || j <= tok);
        const float p = ok ? exp2f(sc[m] * sl2 - lse2) : 0.f;
        Ss[r * kPStride + x + 4 * m] = p * (dp[m] - dlt);
      }
      __syncthreads();
      accumulate<D>(acc, Ss, Ks, r, x);
    }
  }
  if (rvalid) {
    Tin *row = dq + (size_t(tok) * s.Hq + head) * D + 4 * x;
    const float sc = s.scale;
#pragma unroll
    for (int i = 0; i < D / 16; ++i)
      store4(row + 16 * i, make_float4(acc[i].x * sc, acc[i].y * sc, acc[i].z * sc, acc[i].w * sc));
  }
}

// -------------------------------------------------------- backward: dK, dV
template <typename Tin, int D>
__global__ void __launch_bounds__(kThreads) dkdv_kernel(PlanDev plan, AttnShape s, const Tin *__restrict__ q,
                                                        const Tin *__restrict__ k, const Tin *__restrict__ v,
                                                        const Tin *__restrict__ d_o, const float *__restrict__ lse,
                                                        const float *__restrict__ delta, Tin *__restrict__ dk,
                                                        Tin *__restrict__ dv, int32_t *d_status) {
  extern __shared__ float smem[];
  float *Ks = smem;                       // [64][D+4]
  float *Vs = Ks + kRows * (D + 4);       // [64][D+4]
  float *Qs = Vs + kRows * (D + 4);       // [32][D+4]
  float *dOs = Qs + kCols * (D + 4);      // [32][D+4]
  float *Pt = dOs + kCols * (D + 4);      // [64][33]
  float *dSt = Pt + kRows * kPStride;     // [64][33]
  float *rowstat = dSt + kRows * kPStride;  // lse2[32], delta[32]

  const int g = blockIdx.x / plan.n_bwd;
  const int *blk = plan.bwd + 5 * (blockIdx.x % plan.n_bwd);
  const int k0 = blk[1], k1 = blk[2], qb = blk[3], qe = blk[4];
  const int G = s.G, T = s.T;
  if (!range_ok(k0, k1, T) || !range_ok(qb, qe, T) || qb > k0) {
    if (threadIdx.x == 0) flag(d_status, SP_DEV_BAD_PLAN);
    return;
  }
  const int kk0 = k0 + blockIdx.y * kRows;
  if (kk0 >= k1) return;
  const int kk1 = min(k1, kk0 + kRows);
  auto key_src = [&](int c, int &t_, int &h_) {
    t_ = kk0 + c < kk1 ? kk0 + c : -1;
    h_ = g;
  };
  stage_rows<Tin, D>(Ks, k, kRows, s.Hkv, key_src);
  stage_rows<Tin, D>(Vs, v, kRows, s.Hkv, key_src);

  const int c = threadIdx.x >> 2, x = threadIdx.x & 3;
  const int j = kk0 + c;
  const float sl2 = s.scale * kLog2e;
  const int qc = kCols / G;  // query tokens per step
  float4 dka[D / 16], dva[D / 16];
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
    dka[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    dva[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // queries before kk0 cannot see any key of this block
  for (int qt = qb + ((kk0 - qb) / qc) * qc; qt < qe; qt += qc) {
    __syncthreads();
    auto qrow = [&](int r, int &tok, int &head) {
      tok = qt + r / G < qe ? qt + r / G : -1;
      head = g * G + r % G;
    };
    stage_rows<Tin, D>(Qs, q, kCols, s.Hq, qrow);
    stage_rows<Tin, D>(dOs, d_o, kCols, s.Hq, qrow);
    if (threadIdx.x < kCols) {
      const int tk = qt + threadIdx.x / G, hd = g * G + threadIdx.x % G;
      rowstat[threadIdx.x] = tk < qe ? lse[size_t(hd) * T + tk] * kLog2e : 0.f;
      rowstat[kCols + threadIdx.x] = tk < qe ? delta[size_t(hd) * T + tk] : 0.f;
    }
    __syncthreads();
    float st[8], dpt[8];
    scores<D>(Ks, Qs, c, x, st);
    scores<D>(Vs, dOs, c, x, dpt);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int rq = x + 4 * m;
      const int tk = qt + rq / G;
      const bool ok = j < kk1 && tk < qe && j <= tk;
      const float p = ok ? exp2f(st[m] * sl2 - rowstat[rq]) : 0.f;
      Pt[c * kPStride + rq] = p;
      dSt[c * kPStride + rq] = p * (dpt[m] - rowstat[kCols + rq]);
    }
    __syncthreads();
    accumulate<D>(dva, Pt, dOs, c, x);
    accumulate<D>(dka, dSt, Qs, c, x);
  }
  if (j < kk1) {
    const size_t off = (size_t(j) * s.Hkv + g) * D + 4 * x;
    const float sc = s.scale;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      store4(dk + off + 16 * i, make_float4(dka[i].x * sc, dka[i].y * sc, dka[i].z * sc, dka[i].w * sc));
      store4(dv + off + 16 * i, dva[i]);
    }
  }
}

template <int D>
constexpr size_t fwd_smem() {
  return sizeof(float) * (kRows * (D + 4) + 2 * kCols * (D + 4) + kRows * kPStride);
}
template <int D>
constexpr size_t dq_smem() {
  return sizeof(float) * (2 * kRows * (D + 4) + 2 * kCols * (D + 4) + kRows * kPStride);
}
template <int D>
constexpr size_t dkdv_smem() {
  return sizeof(float) * (2 * kRows * (D + 4) + 2 * kCols * (D + 4) + 2 * kRows * kPStride + 2 * kCols);
}

template <typename Tin, int D>
int launch_fwd(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, void *o,
               float *lse, int32_t *d_status, cudaStream_t st) {
  auto kern = fwd_kernel<Tin, D>;
  constexpr size_t smem = fwd_smem<D>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return SP_ERR_CUDA;
  dim3 grid(unsigned(p.n_tiles) * unsigned(s.Hkv), unsigned((p.tile_tokens * s.G + kRows - 1) / kRows));
  kern<<<grid, kThreads, smem, st>>>(p, s, (const Tin *)q, (const Tin *)k, (const Tin *)v, (Tin *)o, lse, d_status);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

template <typename Tin, int D>
int launch_bwd(const PlanDev &p, const AttnShape &s, const void *q, const void *k, const void *v, const void *o,
               const float *lse, const void *d_o, void *dq, void *dk, void *dv, float *delta, int32_t *d_status,
               cudaStream_t st) {
  const long rows = long(s.T) * s.Hq;
  const int dgrid = int(std::min<long>((rows + 7) / 8, 152L * 16));
  delta_kernel<Tin, D><<<dgrid, kThreads, 0, st>>>(s, (const Tin *)o, (const Tin *)d_o, delta);
  if (cudaGetLastError() != cudaSuccess) return SP_ERR_CUDA;

  auto kq = dq_kernel<Tin, D>;
  constexpr size_t sq = dq_smem<D>();
  if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sq)) != cudaSuccess)
    return SP_ERR_CUDA;
  dim3 gq(unsigned(p.n_tiles) * unsigned(s.Hkv), unsigned((p.tile_tokens * s.G + kRows - 1) / kRows));
  kq<<<gq, kThreads, sq, st>>>(p, s, (const Tin *)q, (const Tin *)k, (const Tin *)v, (const Tin *)d_o, lse, delta,
                               (Tin *)dq, d_status);
  if (cudaGetLastError() != cudaSuccess) return SP_ERR_CUDA;

  auto kk = dkdv_kernel<Tin, D>;
  constexpr size_t sk = dkdv_smem<D>();
  if (cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sk)) != cudaSuccess)
    return SP_ERR_CUDA;
  dim3 gk(unsigned(p.n_bwd) * unsigned(s.Hkv), unsigned((p.kv_block + kRows - 1) / kRows));
  kk<<<gk, kThreads, sk, st>>>(p, s, (const Tin *)q, (const Tin *)k, (const Tin *)v, (const Tin *)d_o, lse, delta,
                               (Tin *)dk, (Tin *)dv, d_status);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

}  // namespace

int simt_fwd(const PlanDev &p, const AttnShape &s, int32_t dtype, const void *q, const void *k, const void *v,
             void *o, float *lse, int32_t *d_status, void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == SP_F32)
    return s.D == 64 ? launch_fwd<float, 64>(p, s, q, k, v, o, lse, d_status, st)
                     : launch_fwd<float, 128>(p, s, q, k, v, o, lse, d_status, st);
  return s.D == 64 ? launch_fwd<__nv_bfloat16, 64>(p, s, q, k, v, o, lse, d_status, st)
                   : launch_fwd<__nv_bfloat16, 128>(p, s, q, k, v, o, lse, d_status, st);
}

int simt_bwd(const PlanDev &p, const AttnShape &s, int32_t dtype, const void *q, const void *k, const void *v,
             const void *o, const float *lse, const void *d_o, void *dq, void *dk, void *dv, float *delta,
             int32_t *d_status, void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == SP_F32)
    return s.D == 64 ? launch_bwd<float, 64>(p, s, q, k, v, o, lse, d_o, dq, dk, dv, delta, d_status, st)
                     : launch_bwd<float, 128>(p, s, q, k, v, o, lse, d_o, dq, dk, dv, delta, d_status, st);
  return s.D == 64 ? launch_bwd<__nv_bfloat16, 64>(p, s, q, k, v, o, lse, d_o, dq, dk, dv, delta, d_status, st)
                   : launch_bwd<__nv_bfloat16, 128>(p, s, q, k, v, o, lse, d_o, dq, dk, dv, delta, d_status, st);
}

}  // namespace spc
