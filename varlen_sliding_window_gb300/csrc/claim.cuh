// Run-time work claiming for the backward passes.
//
// Instead of dealing every CTA a fixed share of the longest-first unit list,
// one CTA writes the whole list to the workspace and every CTA claims the
// next unit from a global counter when it is ready for it.  CTAs that start
// late (the dQ pass starts on the SMs the dK/dV pass frees, one by one) or
// whose units turn out slower simply claim fewer units, so the pass ends
// when its work runs out rather than when its most loaded CTA finishes.
// The result does not depend on which CTA takes which unit: no pass
// reduces across units except the dK/dV chains, whose sums run in a fixed
// order.
//
// Per pass, four words in the workspace:
//   [0] state: idle -> planning (one CTA won the election) -> list ready, or
//       fixed shares when the list does not fit (every CTA then plans its
//       own share as before)
//   [1] next unit to hand out   [2] CTAs finished   [3] number of units
// The preprocess zeroes them, and the last CTA of a pass to finish resets
// them, so a pass can also run again on the same workspace.
#pragma once
#include <cstdint>

#include "ptx.cuh"
#include "sched.cuh"

namespace vsw {

enum : int { kClaimIdle = 0, kClaimPlanning = 1, kClaimReady = 2, kClaimFixed = 3 };

// Thread 0 of a CTA: true if this CTA is the one that writes the list.
__device__ __forceinline__ bool claim_elect(int* words) {
  return atomicCAS(&words[0], kClaimIdle, kClaimPlanning) == kClaimIdle;
}

// Thread 0 of the planning CTA, after every thread's list writes are fenced
// and a CTA barrier: n >= 0 units are ready, n < 0 means fixed shares.
__device__ __forceinline__ void claim_publish(int* words, int n) {
  if (n >= 0) words[3] = n;
  __threadfence();
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(words), "r"(n >= 0 ? kClaimReady : kClaimFixed)
               : "memory");
}

// Thread 0: waits (bounded) until the list is ready or fixed shares are
// decided; returns the state, or -1 if the wait gave up (the status word then
// holds the timeout and the CTA's abort flag is set).
__device__ __forceinline__ int claim_wait(int* words, volatile int* abort_flag, int* status) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(words) : "memory");
    if (v == kClaimReady || v == kClaimFixed) return v;
    if (global_timer_ns() - t0 > VSW_WAIT_TIMEOUT_NS) {
      *abort_flag = 1;
      if (status) atomicExch(status, kDevTimeout);
      return -1;
    }
    __nanosleep(128);
  }
}

// The next unit (global position) for this CTA.
__device__ __forceinline__ int claim_next(int* words) { return atomicAdd(&words[1], 1); }

// A unit of the published list, read from L2 (the list changes from call to
// call at the same address, so no stale L1 copy may be used).
__device__ __forceinline__ WorkItem claim_item(const WorkItem* list, int u) {
  const int* src = reinterpret_cast<const int*>(list + u);
  WorkItem w;
  w.seg_lo = __ldcg(src + 0);
  w.seg_hi = __ldcg(src + 1);
  w.blk = __ldcg(src + 2);
  w.unit = __ldcg(src + 3);
  w.t0 = __ldcg(src + 4);
  w.t1 = __ldcg(src + 5);
  w.chain = __ldcg(src + 6);
  w.link = __ldcg(src + 7);
  w.order = __ldcg(src + 8);
  return w;
}

// Thread 0, once per CTA at the end of the kernel: the last CTA to finish
// resets the words for the next run.
__device__ __forceinline__ void claim_finish(int* words) {
  __threadfence();
  if (atomicAdd(&words[2], 1) == (int)gridDim.x - 1) {
    words[1] = 0;
    words[2] = 0;
    words[3] = 0;
    __threadfence();
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(words), "r"(kClaimIdle) : "memory");
  }
}

}  // namespace vsw
