// Longest-first tile scheduler, computed on the device from cu_seqlens.
//
// Work is split into 128-token tiles aligned to each segment's start.  The
// cost of a q tile (forward, dQ pass) is the number of kv tiles it sees,
// which depends only on the tile's index b inside its segment and grows with
// b; the cost of a kv tile (dK/dV pass) is the number of q tiles that see it,
// which grows with the tile's distance from the segment's end.  Visiting
// "levels" from the largest index down therefore yields the work in
// longest-first (LPT) order without sorting: level L holds one item per
// segment that has more than L tiles.
//
// Every item expands to `units_per_item` units (heads or head groups).  Unit
// u goes to CTA  pos  in round  r = u / G  with  pos = u % G  on even rounds
// and G-1-pos on odd rounds (a snake order that evens out the per-CTA cost).
// Each CTA enumerates the order itself and keeps only its own units, so no
// global workspace and no host synchronisation are needed.
#pragma once
#include <cstdint>

#include "mask.cuh"

namespace vsw {

struct WorkItem {
  int seg_lo;
  int seg_hi;
  int blk;   // tile index inside the segment
  int unit;  // head / head-group index
};

constexpr int kMaxItemsPerCta = 64;

// Called by one full warp.  cu (shared memory) holds nseg+1 boundaries.
// reverse == false: level L -> tile L        (q tiles: forward, dQ)
// reverse == true : level L -> tile nblk-1-L (kv tiles: dK/dV)
// Returns the number of items written (or -1 if more than max_out).
__device__ __forceinline__ int build_schedule(const int* cu, int nseg, int max_levels, int units_per_item,
                                              bool reverse, WorkItem* out, int max_out, int* counter, int cta,
                                              int G) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) *counter = 0;
  __syncwarp();
  int base = 0;  // items enumerated so far (global order)
  bool overflow = false;
  for (int lvl = max_levels - 1; lvl >= 0; --lvl) {
    for (int s0 = 0; s0 < nseg; s0 += 32) {
      const int s = s0 + lane;
      int lo = 0, hi = 0, nb = 0;
      if (s < nseg) {
        lo = cu[s];
        hi = cu[s + 1];
        nb = num_tiles(hi - lo);
      }
      const bool has = s < nseg && nb > lvl;
      const unsigned m = __ballot_sync(0xffffffffu, has);
      if (has) {
        const int p = base + __popc(m & ((1u << lane) - 1u));
        for (int h = 0; h < units_per_item; ++h) {
          const long long u = (long long)p * units_per_item + h;
          const long long r = u / G;
          const int pos = (int)(u - r * G);
          const int owner = (r & 1) ? (G - 1 - pos) : pos;
          if (owner == cta) {
            const int slot = atomicAdd(counter, 1);
            if (slot < max_out) {
              out[slot].seg_lo = lo;
              out[slot].seg_hi = hi;
              out[slot].blk = reverse ? (nb - 1 - lvl) : lvl;
              out[slot].unit = h;
            } else {
              overflow = true;
            }
          }
        }
      }
      base += __popc(m);
    }
  }
  __syncwarp();
  overflow = __any_sync(0xffffffffu, overflow);
  const int n = *counter;
  return overflow ? -1 : n;
}

}  // namespace vsw
