// Backward entry point for callers that cannot allocate device memory.
//
// sp_tree_attn_bwd needs a caller-provided device workspace (Delta and, for
// bf16, the fp32 dQ accumulator).  Some callers have no way to provide one:
// code that runs where cudaMalloc is not allowed (a memory pool that owns the
// whole device and forbids other allocations, a runtime that fixes its
// device footprint at start-up, a plugin handed only its input and output
// buffers).  This variant uses a fixed scratch array that belongs to the
// library's own device code, so it performs no allocation call of its own.
//
// The scratch is one file-scope __device__ array of SP_NOALLOC_SCRATCH_BYTES
// on every GPU where the library's device code is loaded, held until the
// process exits.  When that memory is committed depends on CUDA's module
// loading: with the default lazy loading the driver loads this file's device
// code, and commits the 64 MiB, at the first cudaGetSymbolAddress on each
// device -- that is, during the first call of this entry point there; with
// CUDA_MODULE_LOADING=EAGER it is committed when the library's device code is
// loaded into the context.  A caller whose memory pool will take the whole
// device must therefore make one call (or set EAGER) before the pool takes
// it, and before any stream capture.
//
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress (with
// that device current) and caches it together with the device's current
// context: if the context is replaced (after cudaDeviceReset, for example)
// the next call looks the address up again instead of using a stale one.
// All calls on one device share the array: calls whose work overlaps on that
// GPU (for example on two streams) race on it, so the caller must serialise
// them.  Each call rewrites everything it reads from the scratch (Delta is
// recomputed and the dQ accumulator zeroed inside).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = SP_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

std::mutex g_mu;
void *g_addr[kMaxDevices] = {};
CUcontext g_ctx[kMaxDevices] = {};

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of g_bwd_scratch on the current device, looked up once per
// (device, context).  Before the runtime has made the device's context
// current, cuCtxGetCurrent reports none; the lookup then happens (it makes the
// primary context current) and the context is read again for the cache key.
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SP_ERR_CUDA;
  CtxGetCurrentFn get = ctx_get_current();
  if (!get) return SP_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!ctx || !g_addr[dev] || g_ctx[dev] != ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return SP_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return SP_ERR_CUDA;
    g_addr[dev] = p;
    g_ctx[dev] = ctx;
  }
  *out = g_addr[dev];
  return SP_OK;
}

}  // namespace

extern "C" int sp_tree_attn_bwd_noalloc(const sp_plan *plan, int32_t dtype, const void *q, const void *k,
                                        const void *v, const void *o, const float *lse, const void *d_o, void *dq,
                                        void *dk, void *dv, int32_t T, int32_t Hq, int32_t Hkv, int32_t D,
                                        float softmax_scale, int32_t *d_status, void *stream) {
  if (sp_tree_attn_bwd_workspace_bytes(dtype, T, Hq, D) > kScratchBytes) return SP_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (T > 0) {
    if (int rc = scratch_address(&scratch)) return rc;
  }
  return sp_tree_attn_bwd(plan, dtype, q, k, v, o, lse, d_o, dq, dk, dv, scratch, kScratchBytes, T, Hq, Hkv, D,
                          softmax_scale, d_status, stream);
}
