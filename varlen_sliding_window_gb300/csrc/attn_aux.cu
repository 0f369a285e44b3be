// Small kernels around the attention passes: the backward preprocess
// D = rowsum(dout * out) and the mask-range test hook.
#include <cuda_bf16.h>

#include "attn_internal.h"
#include "mask.cuh"

namespace vsw {

namespace {

// D[h, i] = sum_c dout[i,h,c] * out[i,h,c]  (fp32 accumulation of bf16 values).
// 16 threads per (token, head) row, each reading 16 contiguous bytes of both
// tensors; rows are visited in memory order so loads are fully coalesced.
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const uint4* __restrict__ dout,
                                                             const uint4* __restrict__ out,
                                                             float* __restrict__ delta, int total, int hq) {
  const long long rows = (long long)total * hq;
  const int sub = threadIdx.x & 15;
  // The loop bound is warp-uniform (a warp covers two consecutive rows) so that
  // the shuffles below always see both half-warps.
  for (long long r0 = (long long)blockIdx.x * 16 + ((threadIdx.x >> 5) << 1); r0 < rows;
       r0 += (long long)gridDim.x * 16) {
    const long long r = r0 + ((threadIdx.x >> 4) & 1);
    const bool valid = r < rows;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const uint4 a = valid ? dout[r * 16 + sub] : zero;
    const uint4 b = valid ? out[r * 16 + sub] : zero;
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = __bfloat1622float2(a2[e]);
      const float2 y = __bfloat1622float2(b2[e]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (sub == 0 && valid) {
      const int i = (int)(r / hq), h = (int)(r % hq);
      delta[(size_t)h * total + i] = acc;
    }
  }
}

__device__ int find_segment(const int* cu, int nseg, int i) {
  // largest s with cu[s] <= i (then cu[s+1] > i because cu is non-decreasing
  // and the largest such s skips empty segments)
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= i) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void mask_probe_kernel(const int* __restrict__ cu, int nseg, int total, int window, int max_levels,
                                  int by_key, int* __restrict__ ranges) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= total) return;
  const int s = find_segment(cu, nseg, x);
  const int lo = cu[s], hi = cu[s + 1];
  int first = 0, last = -1, count = 0;
  auto add = [&](int a, int b) {  // tokens [a, b], a <= b
    if (count == 0 || a < first) first = a;
    if (b > last) last = b;
    count += b - a + 1;
  };
  if (!by_key) {
    // Query x, as the forward / dQ kernels visit it.
    const int b = (x - lo) / kTile;
    if (b < max_levels) {
      const int q0 = lo + b * kTile;
      for (int n = first_kv_tile(b, window); n <= b; ++n) {
        const int k0 = lo + n * kTile;
        int c0 = 0, c1 = kTile - 1;
        if (!tile_fully_visible(q0, k0, window)) {
          row_visible_cols(x, k0, window, c0, c1);
          c0 = max(c0, 0);
          c1 = min(c1, kTile - 1);
        }
        if (c0 <= c1) add(k0 + c0, k0 + c1);
      }
    }
  } else {
    // Key x, as the dK/dV kernel visits it.
    const int nb = num_tiles(hi - lo);
    const int n = (x - lo) / kTile;
    if (nb - 1 - n < max_levels) {
      const int k0 = lo + n * kTile;
      const int bl = last_q_tile(n, nb, window);
      for (int b = n; b <= bl; ++b) {
        const int q0 = lo + b * kTile;
        int c0 = 0, c1 = kTile - 1;
        if (!tile_fully_visible_kv(k0, q0, hi, window)) {
          col_visible_rows(x, q0, hi, window, c0, c1);
          c0 = max(c0, 0);
          c1 = min(c1, kTile - 1);
        }
        if (c0 <= c1) add(q0 + c0, q0 + c1);
      }
    }
  }
  ranges[3 * x + 0] = count ? first : 0;
  ranges[3 * x + 1] = count ? last : -1;
  ranges[3 * x + 2] = count;
}

}  // namespace

int launch_bwd_preprocess(const BwdParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.a.total * p.a.hq;
  long long blocks = (rows + 15) / 16;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  bwd_preprocess_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const uint4*>(p.dout),
                                                              static_cast<const uint4*>(p.out), p.delta,
                                                              p.a.total, p.a.hq);
  return (int)cudaGetLastError();
}

int launch_mask_probe(const int* cu_seqlens, int nseg, int total, int window, int max_levels, int by_key,
                      int* ranges, cudaStream_t stream) {
  mask_probe_kernel<<<(total + 255) / 256, 256, 0, stream>>>(cu_seqlens, nseg, total, window, max_levels, by_key,
                                                              ranges);
  return (int)cudaGetLastError();
}

}  // namespace vsw
