// Small kernels around the attention passes: the backward preprocess
// D = rowsum(dout * out) and the mask-range test hook.
#include <cuda_bf16.h>

#include "attn_internal.h"
#include "mask.cuh"
#include "ptx.cuh"

namespace vsw {

namespace {

// D[h, i] = sum_c dout[i,h,c] * out[i,h,c]  (fp32 accumulation of bf16 values).
// 16 threads per (token, head) row, each reading 16 contiguous bytes of both
// tensors; a block covers 64 consecutive rows per step (4 rows per thread,
// all 8 loads issued before any arithmetic) so loads are coalesced and many
// are in flight.  HBM-bound: 2 x 256 bytes read + 4 bytes written per row.
// out is read with an evict-first hint (nothing reads it again); dout stays
// cached for the dK/dV and dQ passes that follow.
constexpr int kPreRowsPerBlock = 64;

template <bool DENSE>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const uint4* __restrict__ dout,
                                                             const uint4* __restrict__ out,
                                                             float* __restrict__ delta, int total, int hq,
                                                             RowStrides dout_st, RowStrides out_st,
                                                             int* __restrict__ chain_progress, int nprogress) {
  grid_dependency_wait();
  // The passes that follow count chain arrivals and claimed units from zero;
  // block 0 clears the counters before it lets the next kernel start (the
  // planning kernel of the backward sets the claim words right away).
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < nprogress; e += blockDim.x) chain_progress[e] = 0;
    __threadfence();
    __syncthreads();
  }
  // Everything before this kernel is complete: the next kernel may start
  // (it waits for this one before reading what it writes).
  grid_dependents_launch();
  const long long rows = (long long)total * hq;
  const int sub = threadIdx.x & 15;
  const int r_in = threadIdx.x >> 4;  // 0..15
  for (long long base = (long long)blockIdx.x * kPreRowsPerBlock; base < rows;
       base += (long long)gridDim.x * kPreRowsPerBlock) {
    uint4 a[4], b[4];
    bool valid[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const long long r = base + 16 * k + r_in;
      valid[k] = r < rows;
      // Row r = (token i, head h); offsets in 16-byte units.  Dense tensors
      // (the usual case) need no division.
      long long od = r * 16, oo = r * 16;
      if (!DENSE) {
        const long long i = r / hq, h = r - i * hq;
        od = (i * dout_st.token + h * dout_st.head) / 8;
        oo = (i * out_st.token + h * out_st.head) / 8;
      }
      a[k] = valid[k] ? __ldg(dout + od + sub) : make_uint4(0, 0, 0, 0);
      b[k] = valid[k] ? __ldcs(out + oo + sub) : make_uint4(0, 0, 0, 0);
    }
    float acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[k]);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b[k]);
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(a2[e]);
        const float2 y = __bfloat1622float2(b2[e]);
        s = fmaf(x.x, y.x, s);
        s = fmaf(x.y, y.y, s);
      }
      acc[k] = s;
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
    if (sub == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (!valid[k]) continue;
        const long long r = base + 16 * k + r_in;
        const int i = (int)(r / hq), h = (int)(r % hq);
        delta[(size_t)h * total + i] = acc[k];
      }
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
  long long blocks = (rows + kPreRowsPerBlock - 1) / kPreRowsPerBlock;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  const bool dense = p.dout_st.token == 128LL * p.a.hq && p.dout_st.head == 128 &&
                     p.out_st.token == 128LL * p.a.hq && p.out_st.head == 128;
  return (int)launch_pdl(dense ? bwd_preprocess_kernel<true> : bwd_preprocess_kernel<false>, dim3((unsigned)blocks),
                         dim3(256), 0, stream,
                         static_cast<const uint4*>(p.dout), static_cast<const uint4*>(p.out), p.delta, p.a.total,
                         p.a.hq, p.dout_st, p.out_st, p.chain_progress, p.chain_progress ? kProgressInts : 0);
}

int launch_mask_probe(const int* cu_seqlens, int nseg, int total, int window, int max_levels, int by_key,
                      int* ranges, cudaStream_t stream) {
  mask_probe_kernel<<<(total + 255) / 256, 256, 0, stream>>>(cu_seqlens, nseg, total, window, max_levels, by_key,
                                                              ranges);
  return (int)cudaGetLastError();
}

}  // namespace vsw
