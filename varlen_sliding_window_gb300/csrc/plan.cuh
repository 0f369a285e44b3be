// Work planner run by every thread of a CTA in the kernel prologue.
//
// Items are the same as in sched.cuh: a stationary 128-token tile (q tile for
// the forward and dQ passes, kv tile for the dK/dV pass) with the range of
// streamed tiles the mask lets it see, split into chunks when it is much
// longer than a CTA's fair share (dK/dV pass only), and expanded into
// `units_per_item` units (heads or head groups).
//
// Units are sorted by size, largest first (a stable counting sort, so every
// CTA derives the same order), then dealt to the G CTAs in a snake: round r
// holds units r G .. r G + G - 1, dealt left to right on even rounds and right
// to left on odd ones.  Each CTA expands only its own units (one per round,
// in increasing global order).  The chunks of a split item are independent:
// each writes its partial sums to a buffer of its own and the last one to
// finish adds them in chunk order (see the dK/dV kernel).
// The dealing rule is the one of the single-warp builder in sched.cuh, but
// every step here runs on all threads of the CTA: the prologue goes from
// thousands of dependent shared-memory steps to a few dozen barriers.
//
// Everything lives in shared memory (the caller's tile region, not yet used).
// When the input does not fit (too many items or chunks for the scratch),
// plan_schedule returns kPlanDoesNotFit and the caller uses the single-warp
// builder of sched.cuh instead.
#pragma once
#include <cstdint>

#include "mask.cuh"
#include "sched.cuh"

namespace vsw {

constexpr int kPlanMaxItems = 4096;   // stationary tiles over all segments
constexpr int kPlanMaxChunks = 8192;  // after splitting
constexpr int kPlanDoesNotFit = -2;

// Shared-memory ints plan_schedule needs for nseg segments, G CTAs and
// `threads` threads (upper bounds for the item and chunk arrays).
__host__ __device__ constexpr int plan_scratch_ints(int nseg, int G, int threads) {
  return 2 * (nseg + 1) + 2 * (kPlanMaxItems + 1) + kPlanMaxChunks + kCostBuckets + 64;
}

namespace plan_detail {

// Exclusive prefix sum over v[0..n) in place (all threads; returns the total).
// `tmp` holds at least threads/32 + 1 ints.
__device__ __forceinline__ int block_exclusive_scan(int* v, int n, int* tmp) {
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const int per = (n + nt - 1) / nt;
  const int b0 = min(n, tid * per), b1 = min(n, b0 + per);
  int sum = 0;
  for (int i = b0; i < b1; ++i) sum += v[i];
  int incl = sum;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int x = lane < nw ? tmp[lane] : 0;
    int wi = x;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) tmp[lane] = wi - x;
    if (lane == 31) tmp[nw] = wi;
  }
  __syncthreads();
  int acc = tmp[warp] + incl - sum;
  for (int i = b0; i < b1; ++i) {
    const int x = v[i];
    v[i] = acc;
    acc += x;
  }
  const int total = tmp[nw];
  __syncthreads();
  return total;
}

__device__ __forceinline__ int block_sum(int x, int* tmp) {
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  if ((threadIdx.x & 31) == 0) tmp[threadIdx.x >> 5] = x;
  __syncthreads();
  int s = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += tmp[w];
  __syncthreads();
  return s;
}

// Sum of x and maximum of y over the block in one pass.  `tmp` holds at
// least 2 * threads/32 ints.
__device__ __forceinline__ void block_sum_max(int x, int y, int* tmp, int& sum, int& mx) {
  for (int o = 16; o > 0; o >>= 1) {
    x += __shfl_xor_sync(0xffffffffu, x, o);
    y = max(y, __shfl_xor_sync(0xffffffffu, y, o));
  }
  const int nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    tmp[threadIdx.x >> 5] = x;
    tmp[nw + (threadIdx.x >> 5)] = y;
  }
  __syncthreads();
  sum = 0;
  mx = 0;
  for (int w = 0; w < nw; ++w) {
    sum += tmp[w];
    mx = max(mx, tmp[nw + w]);
  }
  __syncthreads();
}

__device__ __forceinline__ int block_max(int x, int* tmp) {
  for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
  if ((threadIdx.x & 31) == 0) tmp[threadIdx.x >> 5] = x;
  __syncthreads();
  int s = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s = max(s, tmp[w]);
  __syncthreads();
  return s;
}

// Index of the last entry of the sorted array p[0..n) that is <= x (p[0] <= x).
__device__ __forceinline__ int last_le(const int* p, int n, int x) {
  int a = 0, b = n - 1;
  while (a < b) {
    const int mid = (a + b + 1) >> 1;
    if (p[mid] <= x) a = mid; else b = mid - 1;
  }
  return a;
}

}  // namespace plan_detail

// Called by all threads of the CTA (blockDim.x a multiple of 32, at most
// 1024), with cu_seqlens readable.  Writes this CTA's units to out[0..n) in
// global order and returns n (the same value in every thread), -1 if this
// CTA would get more than max_out units, or kPlanDoesNotFit.
// With all_out set (global memory), it instead writes every unit, in global
// order, to all_out[0..n) and returns n, or kPlanDoesNotFit when n exceeds
// all_max (for kernels whose CTAs claim units from the list at run time).
template <bool KV_STATIONARY>
__device__ __forceinline__ int plan_schedule(const int* cu_seqlens, int nseg, int window, int max_levels,
                                          int units_per_item, int chains_max, WorkItem* out, int max_out,
                                          int* scratch, int scratch_ints, int cta, int G,
                                          WorkItem* all_out = nullptr, int all_max = 0) {
  using namespace plan_detail;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int U = units_per_item;
  if (G < 1 || U < 1 || scratch_ints < plan_scratch_ints(nseg, G, nt)) return kPlanDoesNotFit;
  // ---- shared-memory layout
  int* s_cu = scratch;                          // [nseg + 1]
  int* s_tiles = s_cu + (nseg + 1);             // [nseg + 1] tile prefix
  int* s_cost = s_tiles + (nseg + 1);           // [kPlanMaxItems + 1]
  int* s_sbase = s_cost + (kPlanMaxItems + 1);  // prefix of the chunk counts of split items
  int* s_order = s_sbase + (kPlanMaxItems + 1); // [kPlanMaxChunks] item | chunk << 16
  int* s_base = s_order + kPlanMaxChunks;       // [kCostBuckets] size histogram, then bucket cursors
  int* s_misc = s_base + kCostBuckets;          // [64]: scan scratch

  // ---- 1. boundaries and the tile prefix over segments (one warp while
  // that takes at most 32 segments per lane: fewer barriers)
  for (int s = tid; s <= nseg; s += nt) s_cu[s] = cu_seqlens[s];
  __syncthreads();
  int n_items;
  if (nseg <= 32 * 32) {
    if (warp == 0) {
      const int per = (nseg + 31) / 32;
      const int b0 = min(nseg, lane * per), b1 = min(nseg, b0 + per);
      int sum = 0;
      for (int s = b0; s < b1; ++s) sum += num_tiles(s_cu[s + 1] - s_cu[s]);
      int incl = sum;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int acc = incl - sum;
      for (int s = b0; s < b1; ++s) {
        const int x = num_tiles(s_cu[s + 1] - s_cu[s]);
        s_tiles[s] = acc;
        acc += x;
      }
      if (lane == 31) s_tiles[nseg] = incl;
    }
    __syncthreads();
    n_items = s_tiles[nseg];
  } else {
    for (int s = tid; s < nseg; s += nt) s_tiles[s] = num_tiles(s_cu[s + 1] - s_cu[s]);
    __syncthreads();
    n_items = block_exclusive_scan(s_tiles, nseg, s_misc);
    if (tid == 0) s_tiles[nseg] = n_items;
    __syncthreads();
  }
  if (n_items > kPlanMaxItems) return kPlanDoesNotFit;
  // ---- 2. cost (streamed tiles) of every item
  int my_total = 0, my_max = 0;
  for (int e = tid; e < n_items; e += nt) {
    const int s = last_le(s_tiles, nseg, e);
    const int nb = s_tiles[s + 1] - s_tiles[s];
    const int t = e - s_tiles[s];
    const int lvl = KV_STATIONARY ? nb - 1 - t : t;
    int c = 0;
    if (lvl < max_levels) {
      int r0, r1;
      stream_range<KV_STATIONARY>(t, nb, window, r0, r1);
      c = r1 - r0 + 1;
    }
    s_cost[e] = c;
    my_total += c;
    my_max = max(my_max, c);
  }
  int total_cost, max_cost;
  block_sum_max(my_total, my_max, s_misc, total_cost, max_cost);
  // ---- 3. split limit C (streamed tiles per chunk), as in sched.cuh: every
  // chunk of a split item needs a partial-sum buffer per unit
  int C = 0x7fffffff;
  if (chains_max > 0) {
    const long long avg = ((long long)total_cost * U + G - 1) / G;
    C = max(5, (int)avg);
    while (C < max_cost) {
      int mine = 0;
      for (int e = tid; e < n_items; e += nt) mine += s_cost[e] > C ? (s_cost[e] + C - 1) / C : 0;
      const int nbuf = block_sum(mine, s_misc);
      if ((long long)nbuf * U <= chains_max) break;
      C *= 2;
    }
    if (C >= max_cost) C = 0x7fffffff;
  }
  // ---- 4. chunks per item; the chunks of split items get consecutive
  // buffers (a prefix sum of their chunk counts, only when something is split)
  int my_chunks = 0;
  for (int e = tid; e < n_items; e += nt) {
    const int c = s_cost[e];
    const int k = c == 0 ? 0 : (c <= C ? 1 : (c + C - 1) / C);
    my_chunks += k;
    if (C != 0x7fffffff) s_sbase[e] = k > 1 ? k : 0;
  }
  const int n_chunks = block_sum(my_chunks, s_misc);
  if (C != 0x7fffffff) block_exclusive_scan(s_sbase, n_items, s_misc);
  if (n_chunks > kPlanMaxChunks) return kPlanDoesNotFit;
  // ---- 5. stable counting sort of the chunks by size, largest first.  Equal
  // sizes keep the order (group of 32 items, chunk index, item).
  auto chunk_of = [&](int e, int& k, int& base, int& rem) {
    const int c = s_cost[e];
    k = c == 0 ? 0 : (c <= C ? 1 : (c + C - 1) / C);
    base = k ? c / k : 0;
    rem = k ? c % k : 0;
  };
  if (C == 0x7fffffff && n_items <= nt) {
    // Nothing split and at most one item per thread: each item's position is
    // its rank (larger cost first, then smaller index), counted in one pass
    // over the costs.  Same order as the counting sort below, in a fraction
    // of its barriers and shared-memory steps.
    if (tid < n_items) {
      const int c = s_cost[tid];
      if (c > 0) {
        const int b = bucket_of(c);
        int rank = 0;
        for (int j = 0; j < n_items; ++j) {
          const int bj = bucket_of(s_cost[j]);
          rank += (bj > b) | ((bj == b) & (j < tid));
        }
        s_order[rank] = tid;
      }
    }
  } else {
  for (int b = tid; b < kCostBuckets; b += nt) s_base[b] = 0;
  __syncthreads();
  // Histogram: lanes with the same bucket add once (most items share a few
  // sizes, and one shared-memory atomic per item would serialise on them).
  for (int e0 = tid - lane; e0 < n_items; e0 += nt) {
    const int e = e0 + lane;
    int k = 0, base = 0, rem = 0;
    if (e < n_items) chunk_of(e, k, base, rem);
    int kmax = k;
    for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    for (int i = 0; i < kmax; ++i) {
      const bool has = i < k;
      const int bk = has ? bucket_of(base + (i < rem ? 1 : 0)) : -1;
      const unsigned same = __match_any_sync(0xffffffffu, bk);
      if (has && lane == __ffs(same) - 1) atomicAdd(&s_base[bk], __popc(same));
    }
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive prefix over buckets in descending size order: lane l takes
    // buckets 511 - 16 l down to 496 - 16 l
    constexpr int kPer = kCostBuckets / 32;
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) sum += s_base[kCostBuckets - 1 - (lane * kPer + i)];
    int incl = sum;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int acc = incl - sum;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int b = kCostBuckets - 1 - (lane * kPer + i);
      const int x = s_base[b];
      s_base[b] = acc;
      acc += x;
    }
    __syncwarp();
    // Scatter in (chunk index, item) order: 32 records per step, equal
    // buckets ranked by lane, the bucket cursor advanced by the group leader.
    const unsigned lt_mask = (1u << lane) - 1u;
    auto place = [&](int e, bool has, int i) {
      int bk = -1;
      if (has) {
        int k, base, rem;
        chunk_of(e, k, base, rem);
        bk = bucket_of(base + (i < rem ? 1 : 0));
      }
      const unsigned active = __ballot_sync(0xffffffffu, has);
      const unsigned same = __match_any_sync(0xffffffffu, bk) & active;
      const int pos = has ? s_base[bk] + __popc(same & lt_mask) : 0;
      __syncwarp();
      if (has && (same & lt_mask) == 0) s_base[bk] += __popc(same);
      __syncwarp();
      if (has) s_order[pos] = e | (i << 16);
    };
    for (int e0 = 0; e0 < n_items; e0 += 32) {
      const int e = e0 + lane;
      int k = 0, base, rem;
      if (e < n_items) chunk_of(e, k, base, rem);
      int ks = k;
      for (int o = 16; o > 0; o >>= 1) ks = max(ks, __shfl_xor_sync(0xffffffffu, ks, o));
      for (int i = 0; i < ks; ++i) place(e, i < k, i);
    }
  }
  }
  __syncthreads();  // s_order complete
  // ---- 6. deal: unit u of round r = u / G goes to CTA u % G on even rounds
  // and G - 1 - (u % G) on odd rounds, so this CTA's unit of round r is
  // r G + (r even ? cta : G - 1 - cta); thread r expands it.
  const int n_units = n_chunks * U;
  // Unit u (global position) as a work item.
  auto expand = [&](int u, WorkItem& w) {
    const int pos = u / U, h = u - pos * U;
    const int rec = s_order[pos];
    const int e = rec & 0xFFFF, ci = rec >> 16;
    int k, base, rem;
    chunk_of(e, k, base, rem);
    const int sg = last_le(s_tiles, nseg, e);
    const int nb = s_tiles[sg + 1] - s_tiles[sg];
    const int t = e - s_tiles[sg];
    int r0, r1;
    stream_range<KV_STATIONARY>(t, nb, window, r0, r1);
    w.seg_lo = s_cu[sg];
    w.seg_hi = s_cu[sg + 1];
    w.blk = t;
    w.unit = h;
    w.t0 = r0 + ci * base + min(ci, rem);
    w.t1 = w.t0 + base + (ci < rem ? 1 : 0) - 1;
    // Chain of (item, unit): buffers base .. base + k - 1, one per chunk.
    w.chain = k > 1 ? s_sbase[e] * U + h * k : -1;
    w.link = ci | (k << 16);
    w.order = u;
  };
  if (all_out) {
    if (n_units > all_max) {
      __syncthreads();
      return kPlanDoesNotFit;
    }
    for (int u = tid; u < n_units; u += nt) {
      WorkItem w;
      expand(u, w);
      all_out[u] = w;
    }
    __threadfence();  // visible GPU-wide before the list is published
    __syncthreads();
    return n_units;
  }
  const int rounds = (n_units + G - 1) / G;
  int n_mine = 0;
  for (int r = 0; r < rounds; ++r) {
    const int u = r * G + ((r & 1) ? G - 1 - cta : cta);
    if (u < n_units) n_mine = r + 1;
  }
  if (n_mine > max_out) {
    __syncthreads();
    return -1;
  }
  for (int r = tid; r < n_mine; r += nt) expand(r * G + ((r & 1) ? G - 1 - cta : cta), out[r]);
  __syncthreads();
  return n_mine;
}

}  // namespace vsw
