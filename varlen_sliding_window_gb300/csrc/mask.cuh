// Which keys a query may see, and which 128-token tiles that touches.
//
// Document masking (research.dws.rip/llm/kernels, section 01 "How it was
// measured"): no token attends across its document boundary or its row cut,
// so attention is confined to segments [seg_lo, seg_hi) given by cu_seqlens.
// Within a segment attention is causal; local layers add a left window
// (Fig. 2 "Benchmark setup": a 512-token window).  With window_left = w >= 0,
// query i sees key j iff  seg_lo <= j <= i  and  i - j <= w  (w+1 keys
// including itself); w = -1 means global causal.
//
// Tiles are 128 tokens wide and aligned to the segment start, so tile n of a
// segment covers tokens seg_lo + [128 n, 128 n + 127].
#pragma once
#include <cstdint>

namespace vsw {

constexpr int kTile = 128;  // tokens per q tile and per kv tile
constexpr int kHeadDim = 128;
constexpr int kMaxSegments = 8191;  // cu_seqlens entries staged in shared memory

// Index guard used before every global access that depends on cu_seqlens.
__host__ __device__ __forceinline__ bool token_in_range(int i, int total) { return (unsigned)i < (unsigned)total; }

__host__ __device__ __forceinline__ bool key_visible(int i, int j, int seg_lo, int window_left) {
  return j >= seg_lo && j <= i && (window_left < 0 || i - j <= window_left);
}

__host__ __device__ __forceinline__ int num_tiles(int len) { return (len + kTile - 1) / kTile; }

// KV tiles that q tile b of a segment can see: [first_kv_tile(b), b].
__host__ __device__ __forceinline__ int first_kv_tile(int b, int window_left) {
  if (window_left < 0) return 0;
  const int x = b * kTile - window_left;
  return x <= 0 ? 0 : x / kTile;
}

// Q tiles that can see kv tile n of a segment with `nblk` tiles: [n, last_q_tile(...)].
__host__ __device__ __forceinline__ int last_q_tile(int n, int nblk, int window_left) {
  if (window_left < 0) return nblk - 1;
  const long long x = (long long)n * kTile + (kTile - 1) + window_left;
  const long long t = x / kTile;
  return t < nblk - 1 ? (int)t : nblk - 1;
}

// True when every (query row, key column) pair of the tile pair is visible
// (no per-element mask needed).  q tile rows are tokens q0..q0+127 clipped to
// the segment, kv tile columns k0..k0+127.
__host__ __device__ __forceinline__ bool tile_fully_visible(int q0, int k0, int window_left) {
  // causal: the last key must not exceed the first query
  if (k0 + kTile - 1 > q0) return false;
  // window: the first key must be within w of the last query
  if (window_left >= 0 && (q0 + kTile - 1) - k0 > window_left) return false;
  return true;
}

// Query-stationary view (forward, dQ): query token i against the kv tile
// starting at token k0.  Visible columns c of the tile are lo <= c <= hi.
// Keys before seg_lo never occur (tiles start at the segment start).
__host__ __device__ __forceinline__ void row_visible_cols(int i, int k0, int window_left, int& lo, int& hi) {
  lo = (window_left < 0) ? 0 : i - window_left - k0;
  hi = i - k0;
}

// Key-stationary view (dK/dV): key token j against the q tile starting at
// token q0 of a segment ending at seg_hi.  Visible columns c (query q0 + c)
// are lo <= c <= hi.
__host__ __device__ __forceinline__ void col_visible_rows(int j, int q0, int seg_hi, int window_left, int& lo,
                                                          int& hi) {
  lo = j - q0;
  hi = seg_hi - 1 - q0;
  if (window_left >= 0 && j + window_left - q0 < hi) hi = j + window_left - q0;
}

// Key-stationary: true when every (key row, query column) pair is visible,
// i.e. the q tile lies after the whole kv tile, inside the window of its first
// key, and entirely inside the segment.
__host__ __device__ __forceinline__ bool tile_fully_visible_kv(int k0, int q0, int seg_hi, int window_left) {
  if (q0 < k0 + kTile - 1) return false;
  if (q0 + kTile > seg_hi) return false;
  if (window_left >= 0 && (q0 + kTile - 1) - k0 > window_left) return false;
  return true;
}

}  // namespace vsw
