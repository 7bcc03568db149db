// Bounded mbarrier waits shared by the tensor-core kernels.
#pragma once

#include <cstdint>

#include "../../include/shared_prefix_causal.h"
#include "sm103_ptx.cuh"

namespace spc {

// Polls of one mbarrier before a wait gives up (a few milliseconds to seconds
// of wall time; legitimate waits in these kernels take microseconds).
constexpr uint32_t kSpinLimit = 1u << 22;

// Barrier array base, the CTA's abort flag (shared memory) and the caller's
// status word.  Every wait is bounded: when one expires it sets the abort
// flag and SP_DEV_TIMEOUT; waits elsewhere in the CTA then give up at their
// next check, so the CTA winds down instead of hanging.
struct Ctl {
  uint32_t bar0;
  volatile int *abort;
  int32_t *d_status;
  uint32_t limit = kSpinLimit;
  __device__ uint32_t bar(int i) const { return bar0 + 8u * uint32_t(i); }
  // Bounded wait; false if it expired here or another role gave up first.
  // kCluster: cluster-scope acquire, for barriers the peer CTA of a pair
  // arrives on.
  template <bool kCluster = false>
  __device__ bool wait(int i, uint32_t parity) const {
    for (uint32_t it = 0;; ++it) {
      if (kCluster ? ptx::mbar_try_wait_cluster(bar(i), parity) : ptx::mbar_try_wait(bar(i), parity)) return true;
      if ((it & 255u) == 255u) {
        if (*abort) return false;
        if (it >= limit) {
          *abort = 1;
          if (d_status) atomicOr(d_status, SP_DEV_TIMEOUT);
          return false;
        }
      }
    }
  }
  __device__ bool wait_cluster(int i, uint32_t parity) const { return wait<true>(i, parity); }
  // Same for a whole warp: one lane polls (32 lanes polling one barrier
  // serialise on it and starve the warps that do the work), the others wait
  // at __syncwarp, which also orders their later reads after lane 0's acquire.
  __device__ bool wait_warp(int i, uint32_t parity) const {
    bool r = true;
    if ((threadIdx.x & 31) == 0) r = wait(i, parity);
    __syncwarp();
    return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
  }
  // Bounded wait used while draining after an abort (ignores the flag).
  __device__ void drain(int i, uint32_t parity) const {
    for (uint32_t it = 0; it < limit; ++it)
      if (ptx::mbar_try_wait(bar(i), parity)) return;
  }
};

// Walks a work item's runs of 128-key blocks (entries of 8 int32: kb, count,
// end per tile slot, causal bits, 0) one block at a time.  The caller stops
// after the item's last block; next() never reads past the current run.
struct RunCursor {
  const int32_t *r;  // current run
  int32_t i = 0;     // block within it
  __device__ explicit RunCursor(const int32_t *first) : r(first) {}
  __device__ int32_t kb() const { return r[0] + 128 * i; }
  __device__ int32_t end(int slot) const { return r[2 + slot]; }
  __device__ bool causal(int slot) const { return (r[6] >> slot) & 1; }
  __device__ void next() {
    if (++i == r[1]) {
      r += 8;
      i = 0;
    }
  }
};

// Checks a work item's runs against the tokens [0, T) and the slots present
// (bit s of `present`); returns the number of blocks, or -1 if any run is
// malformed: an empty or out-of-range run, an end below a block it covers or
// past T, a slot read by nothing or by an absent tile.
__device__ inline int64_t check_runs(const int32_t *runs, int32_t n_runs, int32_t T, uint32_t present) {
  int64_t blocks = 0;
  for (int32_t r = 0; r < n_runs; ++r) {
    const int32_t *e = runs + 8 * size_t(r);
    const int64_t kb = e[0], nb = e[1];
    if (nb < 1 || kb < 0 || kb + 128 * (nb - 1) >= T) return -1;
    const int64_t last = kb + 128 * (nb - 1);
    bool any = false;
    for (int s = 0; s < 4; ++s) {
      const int64_t end = e[2 + s];
      if (end == 0) {
        if ((e[6] >> s) & 1) return -1;
        continue;
      }
      if (!((present >> s) & 1) || end <= last || end > T) return -1;
      any = true;
    }
    if (!any) return -1;
    blocks += nb;
  }
  return blocks;
}

// Per-CTA timing record for measurements of a launch's tail: when enabled (a
// non-null buffer), thread 0 of CTA b writes {start ns, end ns, SM id, 0}
// (global timer) to buf[4 b .. 4 b + 3] for b < cap.  Off, it costs a branch.
struct CtaClock {
  unsigned long long *buf = nullptr;
  int32_t cap = 0;
  __device__ static unsigned long long now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
  }
  __device__ unsigned long long begin() const { return buf ? now() : 0ull; }
  __device__ void end(unsigned long long t0) const {
    if (buf && threadIdx.x == 0 && int64_t(blockIdx.x) < cap) {
      uint32_t sm;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
      unsigned long long *r = buf + 4 * size_t(blockIdx.x);
      r[0] = t0;
      r[1] = now();
      r[2] = sm;
      r[3] = 0;
    }
  }
};

}  // namespace spc
