// Run-time work claiming for the backward passes.
//
// Instead of dealing every CTA a fixed share of the longest-first unit list,
// a planning kernel (one CTA, running under the backward's preprocess)
// writes the whole list of each pass to the workspace, and every CTA of the
// pass claims the next unit from a global counter when it is ready for it.
// CTAs that start late (the dQ pass starts on the SMs the dK/dV pass frees,
// one by one) or whose units turn out slower simply claim fewer units, so a
// pass ends when its work runs out rather than when its most loaded CTA
// finishes.  The result does not depend on which CTA takes which unit: no
// pass reduces across units except the dK/dV chains, whose sums run in a
// fixed order.
//
// Per pass, four words in the workspace:
//   [0] state: idle, list ready, or fixed shares (the list did not fit:
//       every CTA then plans its own share)
//   [1] next unit to hand out   [2] CTAs finished   [3] number of units
// The preprocess zeroes them (before it lets the planning kernel start), the
// planning kernel sets them, and the last CTA of a pass to finish sets them
// back to idle, so a pass run without a fresh plan falls back to fixed shares.
#pragma once
#include <cstdint>

#include "ptx.cuh"
#include "sched.cuh"

namespace vsw {

enum : int { kClaimIdle = 0, kClaimReady = 2, kClaimFixed = 3 };

// Thread 0 of the planning kernel, after every thread's list writes are
// fenced and a CTA barrier: n >= 0 units are ready, n < 0 means fixed shares.
__device__ __forceinline__ void claim_init(int* words, int n) {
  words[1] = 0;
  words[2] = 0;
  words[3] = n >= 0 ? n : 0;
  __threadfence();
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(words), "r"(n >= 0 ? kClaimReady : kClaimFixed)
               : "memory");
}

// True if a list is ready for this pass (read after the pass has waited for
// the kernels before it).
__device__ __forceinline__ bool claim_ready(const int* words) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(words) : "memory");
  return v == kClaimReady;
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

// Thread 0, once per CTA at the end of a pass that claimed: the last CTA to
// finish sets the words back to idle.
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
