// Longest-first tile scheduler, computed on the device from cu_seqlens.
//
// Work is split into 128-token tiles aligned to each segment's start.  An
// item is one stationary tile (a q tile for the forward and dQ passes, a kv
// tile for the dK/dV pass) together with the range of streamed tiles the mask
// lets it see (mask.cuh); its cost is the length of that range.
//
// When splitting is allowed (dK/dV pass, enough workspace), an item whose
// range is longer than a limit C is cut into chunks of at most C streamed
// tiles: a kv tile near the start of a long segment is seen by many q tiles
// and would otherwise be one unit much larger than a CTA's fair share.  The
// chunks of an item form a chain: each writes its partial sums to a buffer
// of its own and the last to finish adds them in chunk order (see the dK/dV
// kernel), so results stay bitwise reproducible.  C is the average per-CTA
// cost (at least 5 tiles), doubled until the chunks of the split items fit in
// the available buffers.  (Half the average balanced fixed shares a little
// better, but every chunk costs a partial-sum write and read; with units
// claimed at run time, or the dQ pass filling the SMs this pass leaves idle,
// fewer and longer chunks make the whole backward shorter.)
//
// Every chunk (or unsplit item) expands into `units_per_item` units (heads or
// head groups) of equal cost.  Units are ordered by cost, largest first, with
// a counting sort whose ranks are computed warp-synchronously (so every CTA
// derives the same global order), then dealt to CTAs in a snake: unit u in
// round r = u / G goes to CTA u % G on even rounds and G-1-(u % G) on odd
// rounds.  Each CTA keeps its own units, in global order.
#pragma once
#include <cstdint>

#include "mask.cuh"

namespace vsw {

struct WorkItem {
  int seg_lo;
  int seg_hi;
  int blk;    // stationary tile index inside the segment
  int unit;   // head / head-group index
  int t0;     // first streamed tile (inside the segment)
  int t1;     // last streamed tile
  int chain;  // -1: not split; else the first partial-sum buffer of this (item, unit)
  int link;   // chunk index in the chain (low 16 bits) | number of chunks << 16
  int order;  // global position of the unit (the CTA processes its units in this order)
};

__device__ __forceinline__ int link_index(const WorkItem& w) { return w.link & 0xffff; }
__device__ __forceinline__ int link_count(const WorkItem& w) { return w.link >> 16; }
constexpr int kCostBuckets = 512;  // costs >= 511 tiles share the last bucket
static_assert(kCostBuckets % 32 == 0, "the bucket prefix gives each lane kCostBuckets / 32 buckets");

// Scratch the builder needs in shared memory, in ints: the histogram / bucket
// bases, a few counters, and room to reorder up to `max_out` items.
__host__ __device__ constexpr int sched_scratch_ints(int max_out) {
  return kCostBuckets + 8 + max_out * (int)(sizeof(WorkItem) / sizeof(int));
}

// Full streamed-tile range of stationary tile `t` of a segment with `nb` tiles.
template <bool KV_STATIONARY>
__device__ __forceinline__ void stream_range(int t, int nb, int window, int& r0, int& r1) {
  if (KV_STATIONARY) {
    r0 = t;
    r1 = last_q_tile(t, nb, window);
  } else {
    r0 = first_kv_tile(t, window);
    r1 = t;
  }
}

__device__ __forceinline__ int bucket_of(int cost) { return cost < kCostBuckets - 1 ? cost : kCostBuckets - 1; }

// Enumerates the items of all segments in a flat order (segment by segment,
// tile by tile), 32 per step, one per lane.  `tiles` (shared) holds the
// exclusive prefix of tile counts per segment, tiles[nseg] = total.
__device__ __forceinline__ void item_at(const int* cu, const int* tiles, int nseg, int e, int& lo, int& hi, int& nb,
                                        int& t) {
  int a = 0, b = nseg - 1;  // last segment whose prefix <= e
  while (a < b) {
    const int mid = (a + b + 1) >> 1;
    if (tiles[mid] <= e) a = mid; else b = mid - 1;
  }
  lo = cu[a];
  hi = cu[a + 1];
  nb = tiles[a + 1] - tiles[a];
  t = e - tiles[a];
}

// Called by one full warp.  cu (shared memory) holds nseg+1 boundaries; sm is
// sched_scratch_ints(max_out) + nseg + 1 ints of shared memory.  Returns the
// number of units kept, sorted by global position (or -1 if more than
// max_out).
template <bool KV_STATIONARY>
__device__ __noinline__ int build_schedule(const int* cu, int nseg, int window, int max_levels, int units_per_item,
                                           int chains_max, WorkItem* out, int max_out, int* sm, int cta, int G) {
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  int* hist = sm;                     // [kCostBuckets]
  int* counters = sm + kCostBuckets;  // [0] kept units
  WorkItem* tmp = reinterpret_cast<WorkItem*>(sm + kCostBuckets + 8);
  int* tiles = sm + sched_scratch_ints(max_out);  // [nseg + 1]
  // ---- tile-count prefix over segments (warp scan, 32 segments per step)
  int carry = 0;
  for (int s0 = 0; s0 < nseg; s0 += 32) {
    const int s = s0 + lane;
    const int nb = s < nseg ? num_tiles(cu[s + 1] - cu[s]) : 0;
    int incl = nb;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (s < nseg) tiles[s] = carry + incl - nb;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) tiles[nseg] = carry;
  __syncwarp();
  const int n_items = carry;
  // Cost (streamed tiles) of flat item e; 0 if it lies beyond max_levels.
  auto item_range = [&](int e, int& lo, int& hi, int& t, int& r0, int& r1) -> int {
    int nb;
    item_at(cu, tiles, nseg, e, lo, hi, nb, t);
    const int lvl = KV_STATIONARY ? nb - 1 - t : t;
    if (lvl >= max_levels) return 0;
    stream_range<KV_STATIONARY>(t, nb, window, r0, r1);
    return r1 - r0 + 1;
  };
  // ---- pass 0: total and largest cost (for the split limit)
  int total_cost = 0, max_cost = 0;
  for (int e0 = 0; e0 < n_items; e0 += 32) {
    const int e = e0 + lane;
    int c = 0;
    if (e < n_items) {
      int lo, hi, t, r0, r1;
      c = item_range(e, lo, hi, t, r0, r1);
    }
    total_cost += c;
    max_cost = max(max_cost, c);
  }
  for (int o = 16; o > 0; o >>= 1) {
    total_cost += __shfl_xor_sync(0xffffffffu, total_cost, o);
    max_cost = max(max_cost, __shfl_xor_sync(0xffffffffu, max_cost, o));
  }
  // ---- split limit C (in streamed tiles)
  int C = 0x7fffffff;
  if (chains_max > 0 && units_per_item > 0) {
    const long long avg = ((long long)total_cost * units_per_item + G - 1) / G;  // tiles per CTA
    C = max(5, (int)avg);
    while (C < max_cost) {
      int nbuf = 0;  // chunks of split items
      for (int e0 = 0; e0 < n_items; e0 += 32) {
        const int e = e0 + lane;
        int k = 0;
        if (e < n_items) {
          int lo, hi, t, r0, r1;
          const int c = item_range(e, lo, hi, t, r0, r1);
          k = c > C ? (c + C - 1) / C : 0;
        }
        for (int o = 16; o > 0; o >>= 1) k += __shfl_xor_sync(0xffffffffu, k, o);
        nbuf += k;
      }
      if ((long long)nbuf * units_per_item <= chains_max) break;
      C *= 2;
    }
    if (C >= max_cost) C = 0x7fffffff;
  }
  // ---- pass 1: histogram of chunk costs
  for (int b = lane; b < kCostBuckets; b += 32) hist[b] = 0;
  __syncwarp();
  for (int e0 = 0; e0 < n_items; e0 += 32) {
    const int e = e0 + lane;
    if (e < n_items) {
      int lo, hi, t, r0, r1;
      const int c = item_range(e, lo, hi, t, r0, r1);
      if (c > 0) {
        const int k = c <= C ? 1 : (c + C - 1) / C;
        const int base = c / k, rem = c % k;
        if (rem) atomicAdd(&hist[bucket_of(base + 1)], rem);
        atomicAdd(&hist[bucket_of(base)], k - rem);
      }
    }
  }
  __syncwarp();
  // ---- exclusive prefix over buckets in descending cost order: lane l takes
  // the 16 buckets 511 - 16l down to 496 - 16l, then a warp scan joins them.
  {
    constexpr int kPer = kCostBuckets / 32;
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) sum += hist[kCostBuckets - 1 - (lane * kPer + i)];
    int incl = sum;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int acc = incl - sum;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int b = kCostBuckets - 1 - (lane * kPer + i);
      const int n = hist[b];
      hist[b] = acc;
      acc += n;
    }
    if (lane == 0) counters[0] = 0;
  }
  __syncwarp();
  // ---- pass 2: positions (deterministic ranks), deal units, keep own
  bool overflow = false;
  int split_seen = 0;  // chunks of the split items enumerated so far (same in every lane)
  for (int e0 = 0; e0 < n_items; e0 += 32) {
    const int e = e0 + lane;
    int lo = 0, hi = 0, t = 0, r0 = 0, r1 = -1, k = 0;
    if (e < n_items) {
      const int c = item_range(e, lo, hi, t, r0, r1);
      if (c > 0) k = c <= C ? 1 : (c + C - 1) / C;
    }
    const int c = r1 - r0 + 1;
    const int base = k ? c / k : 0, rem = k ? c % k : 0;
    // First buffer of this lane's item: split items in enumeration order, k
    // buffers per split item and unit.
    const int ks = k > 1 ? k : 0;
    int kincl = ks;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, kincl, o);
      if (lane >= o) kincl += y;
    }
    const int chain_base = (k > 1) ? (split_seen + kincl - ks) * units_per_item : -1;
    split_seen += __shfl_sync(0xffffffffu, kincl, 31);
    int kmax = k;
    for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    int start = r0;
    for (int i = 0; i < kmax; ++i) {
      const bool has = i < k;
      const int size = has ? base + (i < rem ? 1 : 0) : 0;
      const int bk = has ? bucket_of(size) : -1;
      const unsigned active = __ballot_sync(0xffffffffu, has);
      const unsigned same = __match_any_sync(0xffffffffu, bk) & active;
      int pos = 0;
      if (has) pos = hist[bk] + __popc(same & lt_mask);
      __syncwarp();
      if (has && (same & lt_mask) == 0) hist[bk] += __popc(same);  // group leader advances the base
      __syncwarp();
      if (has) {
        // Units pos*U .. pos*U+U-1; unit u goes to CTA (u % G) or G-1-(u % G).
        int u = pos * units_per_item;
        int r = u / G, pcta = u - r * G;
        for (int h = 0; h < units_per_item; ++h) {
          const int owner = (r & 1) ? (G - 1 - pcta) : pcta;
          if (owner == cta) {
            const int slot = atomicAdd(&counters[0], 1);
            if (slot < max_out) {
              WorkItem& w = out[slot];
              w.seg_lo = lo;
              w.seg_hi = hi;
              w.blk = t;
              w.unit = h;
              w.t0 = start;
              w.t1 = start + size - 1;
              w.chain = (k > 1) ? chain_base + h * k : -1;
              w.link = i | (k << 16);
              w.order = u;
            } else {
              overflow = true;
            }
          }
          ++u;
          if (++pcta == G) {
            pcta = 0;
            ++r;
          }
        }
      }
      start += size;
    }
  }
  __syncwarp();
  overflow = __any_sync(0xffffffffu, overflow);
  if (overflow) return -1;
  const int n = counters[0];
  // ---- sort the kept units by global position (ranks, then scatter and copy back)
  for (int e = lane; e < n; e += 32) {
    const int key = out[e].order;
    int rank = 0;
    for (int f = 0; f < n; ++f) rank += out[f].order < key;
    tmp[rank] = out[e];
  }
  __syncwarp();
  for (int e = lane; e < n; e += 32) out[e] = tmp[e];
  __syncwarp();
  return n;
}

}  // namespace vsw
