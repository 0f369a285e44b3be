// Gated DeltaNet and Kimi Delta attention over packed documents
// (gdn_varlen.h, kda_varlen.h): forward and backward.
//
// The recurrence (per head, state H of d_k x d_v = 128 x 128, reset at every
// segment start):
//     e_t = beta_t (v_t - alpha_t H_{t-1}^T k_t),  H_t = alpha_t H_{t-1} + k_t e_t^T,
//     o_t = scale H_t^T q_t,  alpha_t = exp(g_t)
// (Kimi Delta: alpha_t a decay per key channel, applied as Diag(alpha_t)).
// Chunked form, chunks of 64 tokens aligned to each segment's start, gamma_i
// the running sum of g over the chunk and Gamma_ij = exp(gamma_i - gamma_j):
//     A    = strictly-lower( diag(beta) (K K^T) o Gamma ),   Tm = (I + A)^-1
//     W    = Tm diag(beta e^gamma) K,   U = Tm diag(beta) V        (64 x 128 each)
//     E    = U - W H0                                             (the chunk's e_t)
//     O    = scale ( diag(e^gamma) Q H0 + (lower(Q K^T) o Gamma) E )
//     H1   = e^gamma_last H0 + (diag(e^(gamma_last - gamma)) K)^T E
// (unrolling the recurrence over the chunk: e_t depends on the earlier e_j
// of the chunk through A, which the triangular inverse resolves at once).
//
// Forward kernels:
//   gdn_plan_kernel    one CTA: the chunk table (start, length of every
//                      chunk) and the non-empty segments ordered longest first
//   gdn_prep_kernel    one CTA per (chunk, head), all in parallel: A, Tm,
//   (kda_prep_kernel)  W, U and the masked Q K^T o Gamma, written to the
//                      workspace (bf16), and gamma (fp32)
//   gdn_state_kernel   one CTA per (segment, head, 32 value columns):
//                      eight warps carry H (fp32, in registers) across the
//                      segment's chunks and write O; a producer warp loads
//                      the tiles of chunks c+1 and c+2 by TMA while chunk c
//                      computes
// Backward: the same plan, prep and state pass (the state pass storing the
// chunk-start states and E; the saving forward stores them and O at once),
// then gdn_bwd_state_kernel carries the state's gradient back across each
// segment, and per-chunk local passes form the gradients (gdn_bwd_local_h /
// _wy, kda_bwd_local_h / _wy / _exp).
// The products are small (64-row) and run in bf16 on the warp-level tensor
// core instruction (mma.sync m16n8k16, fp32 accumulation): the state pass is
// a dependent chain of 64-row steps whose state lives in registers, where the
// asynchronous 128-row tcgen05 path has nothing to overlap.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "attn_internal.h"
#include "attn_varlen.h"
#include "gdn_varlen.h"
#include "ptx.cuh"

namespace vsw {

namespace {

constexpr int kC = 64;         // chunk length (tokens)
constexpr int kD = 128;        // d_k = d_v
// Kimi Delta: smallest per-token log decay the block-referenced products
// allow (the decay of 15 tokens stays within float range: 15 x 5.8 < 88).
constexpr float kKdaMinLogDecay = -5.8f;
constexpr int kDvb = 32;       // value columns per state CTA
constexpr int kGdnThreads = 256;   // prep CTA
constexpr int kStateThreads = 256; // state CTA
constexpr int kLocalThreads = 512; // local backward CTAs (their output blocks assume 16 warps)
constexpr int kS128 = 136;     // smem row stride (elements) of 128-wide bf16 tiles: 272 B, conflict-free ldmatrix
constexpr int kS64 = 72;       // 64-wide: 144 B
constexpr int kS32 = 40;       // 32-wide: 80 B
constexpr int kSF = 65;        // fp32 64 x 64 tiles
constexpr int kG = 132;        // fp32 64 x 128 tiles (gates, per channel): 16-byte rows
constexpr int kS4 = 68;        // fp32 64 x 64 tiles read as float4 rows

struct GdnParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* g;
  const float* beta;
  const int* cu;
  __nv_bfloat16* o;
  int total, nh, nseg, max_chunks;
  float scale;
  int* status;  // the device status word (Kimi Delta: gates out of range)
  // workspace
  int* hdr;             // [0] chunks, [1] non-empty segments
  int4* chunks;         // [max_chunks] {start token, length, segment, chunk index in segment}
  int4* segs;           // [nseg] by length, longest first: {first chunk, chunks, start token, length}
  __nv_bfloat16* W;     // [T, H, 128]
  __nv_bfloat16* U;     // [T, H, 128]
  __nv_bfloat16* Aqk;   // [max_chunks, H, 64, 64]: lower(Q K^T) o Gamma
  float* gam;           // [H, T]: gamma (running log decay within the chunk)
  // Kimi Delta (a decay per key channel; g is then [T, H, 128]): the state
  // pass reads Q o e^gamma and K o e^(gamma_last - gamma) instead of q and k,
  // and the chunk's total decay e^gamma_last per channel
  __nv_bfloat16* QB;    // [T, H, 128]
  __nv_bfloat16* KC;    // [T, H, 128]
  float* Bc;            // [max_chunks, H, 128]
  float* Xw;            // Kimi Delta backward: X = (I + A)^-1 of every chunk, fp32 [max_chunks, H, 64, 64]
  float* Araw;          //   and sum_c k_ic k_jc e^(gamma_ic - gamma_jc) (j < i), same layout
  float* Nw;            //   lower(scale dO E^T), same layout
  float* Mw;            //   diag(beta) dA, same layout
  float* dQa;           //   the part of dq that needs the states, fp32 [T, H, 128]
  // backward only
  const __nv_bfloat16* dO;  // [T, H, 128]
  __nv_bfloat16* dq;        // [T, H, 128]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dg;                // [T, H]
  float* dbeta;             // [T, H]
  __nv_bfloat16* H0;        // [max_chunks, H, 128, 128]: state at each chunk's start (bf16)
  __nv_bfloat16* dH1;       // [max_chunks, H, 128, 128]: gradient w.r.t. the state at each chunk's end
  __nv_bfloat16* E;         // [T, H, 128]: E of every chunk
  __nv_bfloat16* dE;        // [T, H, 128]: its gradient
  __nv_bfloat16* dW;        // [T, H, 128]: gradient w.r.t. W
  float* dKa;               // [T, H, 128]: the part of dk that needs the states
  float* dgam;              // [H, T]: the part of d gamma that needs the states
};

// ---------------------------------------------------------------- mma.sync
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Fragment addresses (byte address of the row this lane supplies), for a
// row-major bf16 tile at `base` with row stride `ld` elements:
// A operand, 16 x 16 block at (r0, c0) of a row-major M x K tile.
__device__ __forceinline__ uint32_t frag_a(uint32_t base, int ld, int r0, int c0, int lane) {
  return base + 2u * (uint32_t)((r0 + (lane & 15)) * ld + c0 + ((lane >> 4) << 3));
}
// B operand for two n-tiles (n0, n0 + 8), k-block k0, from storage Bt[n][k]
// (non-transposed load); also the A operand from storage At[k][m] (transposed
// load, same lane pattern with (k0, m0) as (row, column)).
__device__ __forceinline__ uint32_t frag_bt(uint32_t base, int ld, int n0, int k0, int lane) {
  return base + 2u * (uint32_t)((n0 + (lane & 7) + ((lane >> 4) << 3)) * ld + k0 + (((lane >> 3) & 1) << 3));
}
// B operand for two n-tiles (n0, n0 + 8), k-block k0, from storage B[k][n]
// (transposed load).
__device__ __forceinline__ uint32_t frag_b(uint32_t base, int ld, int k0, int n0, int lane) {
  return base + 2u * (uint32_t)((k0 + (lane & 15)) * ld + n0 + ((lane >> 4) << 3));
}

// The state passes' stage tiles as TMA writes them: a 64 x 128 bf16 tile is
// two 64-column halves of 64 rows x 128 B (8 KB each, 1024-byte aligned), and
// the 128-byte swizzle stores the 16-byte chunk j of row r at chunk j ^ (r % 8).
// Byte address of element (r, c), c a multiple of 8.
__device__ __forceinline__ uint32_t sw128(uint32_t base, int r, int c) {
  return base + ((uint32_t)(c >> 6) << 13) + ((uint32_t)r << 7) + ((uint32_t)(((c >> 3) & 7) ^ (r & 7)) << 4);
}
// frag_a and frag_bt over such a tile: the same lanes supply the same
// (row, column) as over a row-major tile.  Eight lanes read eight
// consecutive rows of one column chunk, which the swizzle puts in eight
// different bank groups.
__device__ __forceinline__ uint32_t frag_a_sw(uint32_t base, int r0, int c0, int lane) {
  return sw128(base, r0 + (lane & 15), c0 + ((lane >> 4) << 3));
}
__device__ __forceinline__ uint32_t frag_bt_sw(uint32_t base, int n0, int k0, int lane) {
  return sw128(base, n0 + (lane & 7) + ((lane >> 4) << 3), k0 + (((lane >> 3) & 1) << 3));
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Rows [0, len) of a [T, H, 128] bf16 tensor (token t0 on, head h) into a
// 64 x 128 smem tile with row stride kS128; rows >= len become zero.
__device__ __forceinline__ void load_rows128(uint32_t dst, const __nv_bfloat16* src, int t0, int len, int h, int nh,
                                             int tid, int nt) {
  for (int e = tid; e < kC * 16; e += nt) {
    const int r = e >> 4, c = (e & 15) * 8;
    const bool ok = r < len;
    const __nv_bfloat16* s = src + ((size_t)(t0 + (ok ? r : 0)) * nh + h) * kD + c;
    cp_async16(dst + 2u * (uint32_t)(r * kS128 + c), s, ok);
  }
}

// Rows of a chunk that lie inside [0, T) (all of them for a valid boundary list).
__device__ __forceinline__ int chunk_len(const int4& ch, int total) {
  return (ch.x < 0 || ch.x >= total) ? 0 : min(ch.y, total - ch.x);
}

// Chunk ci of a segment entry {first chunk, chunks, start token, length}:
// the {start token, length} that the chunk table holds for chunk first + ci
// (the planner lays a segment's chunks 64 tokens apart from its start), with
// no load from the table.
__device__ __forceinline__ int4 seg_chunk(const int4& sg, int ci) {
  return make_int4(sg.z + ci * kC, min(kC, sg.w - ci * kC), 0, ci);
}

// gamma per channel: the running sum of g down each of the 128 channels of a
// 64 x 128 fp32 tile (row stride kG), in place, by the 512 threads of a local
// CTA.  Each thread sums one 16-row segment of one channel; then every
// segment adds the totals of the segments above it, in order.  The same
// order in every kernel gives every kernel the same bits.  `tot`: 4 x 128
// floats of scratch.  Begins and ends at a barrier of all threads.  kCheck:
// also returns, to every thread, whether any g of the tile is at or below
// kKdaMinLogDecay or NaN (rows past the chunk hold zeros).
template <bool kCheck = false>
__device__ __forceinline__ bool chan_running_sum(float* G, float* tot, int tid) {
  const int c = tid & (kD - 1), sg = tid >> 7;
  const int i0 = 16 * sg;
  float acc = 0.f;
  bool bad = false;
#pragma unroll 4
  for (int i = i0; i < i0 + 16; ++i) {
    const float g = G[i * kG + c];
    if (kCheck) bad |= !(g > kKdaMinLogDecay);
    acc += g;
    G[i * kG + c] = acc;
  }
  tot[sg * kD + c] = acc;
  if (kCheck) bad = __syncthreads_or(bad);
  else __syncthreads();
  if (sg > 0) {
    float off = tot[c];
    for (int s2 = 1; s2 < sg; ++s2) off += tot[s2 * kD + c];
#pragma unroll 4
    for (int i = i0; i < i0 + 16; ++i) G[i * kG + c] += off;
  }
  __syncthreads();
  return bad;
}

// ============================================================== plan
__global__ void __launch_bounds__(256) gdn_plan_kernel(GdnParams p) {
  __shared__ int s_first[1024 + 1];
  __shared__ int s_hist[1024];
  __shared__ int s_tmp[32];
  grid_dependency_wait();
  const int tid = threadIdx.x, nt = blockDim.x;
  // Chunks per segment and their prefix, 1024 segments per round.
  int base_chunk = 0;
  for (int r0 = 0; r0 < p.nseg; r0 += 1024) {
    const int n = min(1024, p.nseg - r0);
    for (int i = tid; i < n; i += nt) {
      const int L = p.cu[r0 + i + 1] - p.cu[r0 + i];
      s_first[i] = (max(L, 0) + kC - 1) / kC;
    }
    __syncthreads();
    if (tid < 32) {
      // exclusive prefix of s_first[0..n) by warp 0
      const int per = (n + 31) / 32, b0 = min(n, tid * per), b1 = min(n, b0 + per);
      int sum = 0;
      for (int i = b0; i < b1; ++i) sum += s_first[i];
      int incl = sum;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      int acc = incl - sum;
      for (int i = b0; i < b1; ++i) {
        const int x = s_first[i];
        s_first[i] = acc;
        acc += x;
      }
      if (tid == 31) s_first[n] = incl;
    }
    __syncthreads();
    for (int i = tid; i < n; i += nt) {
      const int a = p.cu[r0 + i], L = p.cu[r0 + i + 1] - a;
      const int f = base_chunk + s_first[i];
      // (bounds checked against the table, which a boundary list that breaks
      // its rules could otherwise overrun)
      for (int j = 0; j * kC < L && f + j < p.max_chunks; ++j)
        p.chunks[f + j] = make_int4(a + j * kC, min(kC, L - j * kC), r0 + i, j);
    }
    base_chunk += s_first[n];
    __syncthreads();
  }
  // Non-empty segments, longest first: counting sort on the chunk count
  // (capped at 1023; order inside a bucket is free, only the order of the
  // state CTAs depends on it, not any result).
  for (int b = tid; b < 1024; b += nt) s_hist[b] = 0;
  __syncthreads();
  for (int s = tid; s < p.nseg; s += nt) {
    const int L = p.cu[s + 1] - p.cu[s];
    if (L > 0) atomicAdd(&s_hist[min(1023, (L + kC - 1) / kC)], 1);
  }
  __syncthreads();
  if (tid < 32) {
    // descending exclusive prefix: lane l takes buckets 1023 - 32 l down to 992 - 32 l
    int sum = 0;
    for (int i = 0; i < 32; ++i) sum += s_hist[1023 - (tid * 32 + i)];
    int incl = sum;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += y;
    }
    int acc = incl - sum;
    for (int i = 0; i < 32; ++i) {
      const int b = 1023 - (tid * 32 + i);
      const int x = s_hist[b];
      s_hist[b] = acc;
      acc += x;
    }
    if (tid == 31) s_tmp[0] = incl;
  }
  __syncthreads();
  // first chunk of segment s = number of chunks of the segments before it
  int chunk_base = 0;
  for (int r0 = 0; r0 < p.nseg; r0 += 1024) {
    const int n = min(1024, p.nseg - r0);
    // recompute the per-round prefix (s_first was overwritten by later rounds)
    for (int i = tid; i < n; i += nt) {
      const int L = p.cu[r0 + i + 1] - p.cu[r0 + i];
      s_first[i] = (max(L, 0) + kC - 1) / kC;
    }
    __syncthreads();
    if (tid < 32) {
      const int per = (n + 31) / 32, b0 = min(n, tid * per), b1 = min(n, b0 + per);
      int sum = 0;
      for (int i = b0; i < b1; ++i) sum += s_first[i];
      int incl = sum;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      int acc = incl - sum;
      for (int i = b0; i < b1; ++i) {
        const int x = s_first[i];
        s_first[i] = acc;
        acc += x;
      }
      if (tid == 31) s_first[n] = incl;
    }
    __syncthreads();
    for (int i = tid; i < n; i += nt) {
      const int a = p.cu[r0 + i], L = p.cu[r0 + i + 1] - a;
      if (L > 0) {
        const int nch = (L + kC - 1) / kC;
        const int pos = atomicAdd(&s_hist[min(1023, nch)], 1);
        p.segs[pos] = make_int4(chunk_base + s_first[i], nch, a, L);
      }
    }
    chunk_base += s_first[n];
    __syncthreads();
  }
  if (tid == 0) {
    p.hdr[0] = min(base_chunk, p.max_chunks);
    p.hdr[1] = s_tmp[0];
  }
}

// X = (I + A)^-1 for the strictly lower triangular 64 x 64 A (fp32, row
// stride kSF; X with row stride LDX), in 16 x 16 blocks, by all NT threads of the CTA; R
// holds 3 x 256 floats of scratch.  Ends with a CTA barrier.
// Four consecutive floats from shared memory: one 16-byte load where the
// address allows it (rows of a stride that is a multiple of 4), else four.
template <int LDX>
__device__ __forceinline__ void load4_impl(float (&x)[4], const float* src) {
  if constexpr (LDX % 4 == 0) {
    const float4 v = *reinterpret_cast<const float4*>(src);
    x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) x[q] = src[q];
  }
}

template <int LDX = kSF, int NT = kGdnThreads>
__device__ __forceinline__ void wy_inverse(const float* A, float* X, float* R, int tid) {
  // ---- X = (I + A)^-1 (unit lower triangular) in 16 x 16 blocks.
  // Diagonal blocks by forward substitution, one column per thread (the other
  // threads clear the blocks above the diagonal meanwhile):
  //     X_bb[r][c] = [r == c] - sum_{c <= j < r} A_bb[r][j] X_bb[j][c].
  if (tid < 64) {
    const int b = tid >> 4, c = tid & 15, o = 16 * b;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < r; ++j) acc = fmaf(A[(o + r) * kSF + o + j], x[j], acc);
      x[r] = r < c ? 0.f : (r == c ? 1.f : -acc);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) X[(o + r) * LDX + o + c] = x[r];
  } else {
    // blocks (bi, bj) with bi < bj: 6 blocks of 256
    for (int e = tid - 64; e < 6 * 256; e += NT - 64) {
      const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
      const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
      const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
      X[(16 * bi + r) * LDX + 16 * bj + c] = 0.f;
    }
  }
  __syncthreads();
  // Blocks below the diagonal, nearest first (d = i - j = 1, 2, 3):
  //     X_ij = -X_ii R_ij,   R_ij = sum_{j <= k < i} A_ik X_kj
  // (the rows of block i of (I + A) X = I), R_ij kept in R.  Each thread
  // computes four adjacent columns of one row: per k one broadcast element of
  // the left factor and four of the right one, which bounds these products by
  // shared-memory reads less than one element per product did.  Two partial
  // sums per output (k even, odd), added in a fixed order.
  for (int d = 1; d < 4; ++d) {
    const int nb = 4 - d;  // blocks (j + d, j), j = 0 .. nb - 1
    for (int e = tid; e < nb * 64; e += NT) {
      const int j = e >> 6, r = (e >> 2) & 15, c = (e & 3) * 4, i = j + d;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      for (int kb = 16 * j; kb < 16 * i; kb += 16) {
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float a = A[(16 * i + r) * kSF + kb + t];
          float x[4];
          load4_impl<LDX>(x, &X[(kb + t) * LDX + 16 * j + c]);
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[t & 1][q] = fmaf(a, x[q], acc[t & 1][q]);
        }
      }
      *reinterpret_cast<float4*>(&R[(j << 8) + (r << 4) + c]) =
          make_float4(acc[0][0] + acc[1][0], acc[0][1] + acc[1][1], acc[0][2] + acc[1][2], acc[0][3] + acc[1][3]);
    }
    __syncthreads();
    for (int e = tid; e < nb * 64; e += NT) {
      const int j = e >> 6, r = (e >> 2) & 15, c = (e & 3) * 4, i = j + d;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float xa = X[(16 * i + r) * LDX + 16 * i + k];
        const float4 rr = *reinterpret_cast<const float4*>(&R[(j << 8) + (k << 4) + c]);
        acc[k & 1][0] = fmaf(xa, rr.x, acc[k & 1][0]);
        acc[k & 1][1] = fmaf(xa, rr.y, acc[k & 1][1]);
        acc[k & 1][2] = fmaf(xa, rr.z, acc[k & 1][2]);
        acc[k & 1][3] = fmaf(xa, rr.w, acc[k & 1][3]);
      }
      float* xo = &X[(16 * i + r) * LDX + 16 * j + c];
#pragma unroll
      for (int q = 0; q < 4; ++q) xo[q] = -(acc[0][q] + acc[1][q]);
    }
    __syncthreads();
  }
}

// ============================================================== prep
// Shared memory of the prep CTA.  Arrays whose lifetimes do not overlap
// share space, so that three CTAs fit on an SM: X takes Q's place (Q is last
// read by Q K^T, X first written by the inverse, a barrier between them; the
// two have the same size), T1 and T2 take the place of A and R (both last
// read by the inverse, which ends on a barrier).
struct PrepSmem {
  __nv_bfloat16 K[kC * kS128];
  union {
    __nv_bfloat16 Q[kC * kS128];
    float X[kC * kS4];  // (I + A)^-1, fp32 (rows of 16-byte multiples for the inverse's wide reads)
  };
  __nv_bfloat16 V[kC * kS128];
  union {
    struct {
      float A[kC * kSF];              // A, fp32
      alignas(16) float R[3 * 256];  // off-diagonal block products
    } ar;
    struct {
      __nv_bfloat16 T1[kC * kS64];  // X diag(beta e^gamma)
      __nv_bfloat16 T2[kC * kS64];  // X diag(beta)
    } t;
  };
  float gam[kC];
  float bet[kC];
};

static_assert(sizeof(PrepSmem::Q) == sizeof(PrepSmem::X), "X fills Q's place exactly");
static_assert(sizeof(PrepSmem) <= 75 * 1024, "three prep CTAs per SM");

__global__ void __launch_bounds__(kGdnThreads, 3) gdn_prep_kernel(GdnParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  PrepSmem& sm = *reinterpret_cast<PrepSmem*>(smem_raw);
  grid_dependency_wait();
  const int c = blockIdx.x, h = blockIdx.y;
  // (both loads in flight at once: the table entry is in bounds for every
  // c < max_chunks, and ignored past the number of chunks)
  const int n_chunks = __ldcg(p.hdr);
  const int4 ch = p.chunks[c];
  if (c >= n_chunks) return;
  const int t0 = ch.x;
  if (t0 < 0 || t0 >= p.total) return;  // only with a boundary list that breaks its rules
  const int len = min(ch.y, p.total - t0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sK = smem_u32(sm.K), sQ = smem_u32(sm.Q), sV = smem_u32(sm.V);
  load_rows128(sK, p.k, t0, len, h, p.nh, tid, kGdnThreads);
  load_rows128(sQ, p.q, t0, len, h, p.nh, tid, kGdnThreads);
  load_rows128(sV, p.v, t0, len, h, p.nh, tid, kGdnThreads);
  cp_async_commit();
  if (warp == 0) {
    // gamma = running sum of g over the chunk (2 tokens per lane), beta
    const int i0 = 2 * lane;
    const float g0 = i0 < len ? p.g[(size_t)(t0 + i0) * p.nh + h] : 0.f;
    const float g1 = i0 + 1 < len ? p.g[(size_t)(t0 + i0 + 1) * p.nh + h] : 0.f;
    const float s = g0 + g1;
    float incl = s;
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const float ex = incl - s;
    sm.gam[i0] = ex + g0;
    sm.gam[i0 + 1] = ex + g0 + g1;
    sm.bet[i0] = i0 < len ? p.beta[(size_t)(t0 + i0) * p.nh + h] : 0.f;
    sm.bet[i0 + 1] = i0 + 1 < len ? p.beta[(size_t)(t0 + i0 + 1) * p.nh + h] : 0.f;
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- K K^T and Q K^T: warp w takes rows [16 (w % 4), +16) x columns [32 (w / 4), +32).
  const int r0 = 16 * (warp & 3);
  const int c0 = 32 * (warp >> 2);
  float skk[4][4], sqk[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) skk[n][e] = sqk[n][e] = 0.f;
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    uint32_t ak[4], aq[4];
    ldsm_x4(ak, frag_a(sK, kS128, r0, 16 * kk, lane));
    ldsm_x4(aq, frag_a(sQ, kS128, r0, 16 * kk, lane));
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t b[4];
      ldsm_x4(b, frag_bt(sK, kS128, c0 + 16 * np, 16 * kk, lane));
      mma_bf16(skk[2 * np], ak, b[0], b[1]);
      mma_bf16(skk[2 * np + 1], ak, b[2], b[3]);
      mma_bf16(sqk[2 * np], aq, b[0], b[1]);
      mma_bf16(sqk[2 * np + 1], aq, b[2], b[3]);
    }
  }
  // A_ij = beta_i Gamma_ij (k_i . k_j) for j < i; lower(Q K^T) o Gamma (j <= i) to the workspace.
  __nv_bfloat16* aqk = p.Aqk + ((size_t)c * p.nh + h) * (kC * kC);
#pragma unroll
  for (int n = 0; n < 4; ++n) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = r0 + (lane >> 2) + 8 * hr;
      const int j = c0 + 8 * n + 2 * (lane & 3);
      const float gi = sm.gam[i], bi = sm.bet[i];
      const float G0 = j <= i ? __expf(gi - sm.gam[j]) : 0.f;
      const float G1 = j + 1 <= i ? __expf(gi - sm.gam[j + 1]) : 0.f;
      sm.ar.A[i * kSF + j] = j < i ? bi * G0 * skk[n][2 * hr] : 0.f;
      sm.ar.A[i * kSF + j + 1] = j + 1 < i ? bi * G1 * skk[n][2 * hr + 1] : 0.f;
      *reinterpret_cast<uint32_t*>(aqk + i * kC + j) = pack2(G0 * sqk[n][2 * hr], G1 * sqk[n][2 * hr + 1]);
    }
  }
  __syncthreads();
  wy_inverse<kS4, kGdnThreads>(sm.ar.A, sm.X, sm.ar.R, tid);
  // ---- T1 = X diag(beta e^gamma), T2 = X diag(beta) (bf16)
  for (int e = tid; e < kC * kC / 2; e += kGdnThreads) {
    const int i = e >> 5, j = (e & 31) * 2;
    const float x0 = sm.X[i * kS4 + j], x1 = sm.X[i * kS4 + j + 1];
    const float b0 = sm.bet[j], b1 = sm.bet[j + 1];
    *reinterpret_cast<uint32_t*>(&sm.t.T1[i * kS64 + j]) =
        pack2(x0 * b0 * __expf(sm.gam[j]), x1 * b1 * __expf(sm.gam[j + 1]));
    *reinterpret_cast<uint32_t*>(&sm.t.T2[i * kS64 + j]) = pack2(x0 * b0, x1 * b1);
  }
  __syncthreads();
  // ---- W = T1 K, U = T2 V: warp w rows [16 (w % 4), +16) x columns [64 (w / 4), +64).
  const int d0 = 64 * (warp >> 2);
  float cw[8][4], cu[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) cw[n][e] = cu[n][e] = 0.f;
  const uint32_t sT1 = smem_u32(sm.t.T1), sT2 = smem_u32(sm.t.T2);
#pragma unroll
  for (int kk = 0; kk < kC / 16; ++kk) {
    uint32_t a1[4], a2[4];
    ldsm_x4(a1, frag_a(sT1, kS64, r0, 16 * kk, lane));
    ldsm_x4(a2, frag_a(sT2, kS64, r0, 16 * kk, lane));
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t bk[4], bv[4];
      ldsm_x4_t(bk, frag_b(sK, kS128, 16 * kk, d0 + 16 * np, lane));
      ldsm_x4_t(bv, frag_b(sV, kS128, 16 * kk, d0 + 16 * np, lane));
      mma_bf16(cw[2 * np], a1, bk[0], bk[1]);
      mma_bf16(cw[2 * np + 1], a1, bk[2], bk[3]);
      mma_bf16(cu[2 * np], a2, bv[0], bv[1]);
      mma_bf16(cu[2 * np + 1], a2, bv[2], bv[3]);
    }
  }
  __syncthreads();  // K, V, Q no longer read: stage W in K's place, U in V's
#pragma unroll
  for (int n = 0; n < 8; ++n) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = r0 + (lane >> 2) + 8 * hr;
      const int j = d0 + 8 * n + 2 * (lane & 3);
      *reinterpret_cast<uint32_t*>(&sm.K[i * kS128 + j]) = pack2(cw[n][2 * hr], cw[n][2 * hr + 1]);
      *reinterpret_cast<uint32_t*>(&sm.V[i * kS128 + j]) = pack2(cu[n][2 * hr], cu[n][2 * hr + 1]);
    }
  }
  __syncthreads();
  for (int e = tid; e < kC * 16; e += kGdnThreads) {
    const int r = e >> 4, cc = (e & 15) * 8;
    if (r < len) {
      const size_t off = ((size_t)(t0 + r) * p.nh + h) * kD + cc;
      *reinterpret_cast<uint4*>(p.W + off) = *reinterpret_cast<const uint4*>(&sm.K[r * kS128 + cc]);
      *reinterpret_cast<uint4*>(p.U + off) = *reinterpret_cast<const uint4*>(&sm.V[r * kS128 + cc]);
    }
  }
  if (tid < kC && tid < len) p.gam[(size_t)h * p.total + t0 + tid] = sm.gam[tid];
}

// ============================================================== prep, a decay per channel (Kimi Delta)
// As gdn_prep_kernel, with gamma a running sum per key channel (B = e^gamma):
//     A_ij   = beta_i sum_c k_ic k_jc e^(gamma_ic - gamma_jc)   (j < i)
//     Aqk_ij =        sum_c q_ic k_jc e^(gamma_ic - gamma_jc)   (j <= i)
//     W = X diag(beta) (K o B),  U = X diag(beta) V,  X = (I + A)^-1
// and, for the state pass, QB = Q o B, KC = K o e^(gamma_last - gamma) and
// e^gamma_last.  The exponent gamma_i - gamma_j is split at a reference token
// r = the first row of i's 16-row block:
//     e^(gamma_i - gamma_j) = e^(gamma_i - gamma_r) e^(gamma_r - gamma_j),
// so the first factor is at most 1 and the second is at most 1 for j < r and
// at most the decay of 15 tokens (j in i's block); each block of 16 rows of A
// is then one matrix product of scaled operands.  (The decay over 15 tokens
// must stay within float range, e^88: per-token log decays above -5.8.)
struct KdaPrepSmem {
  __nv_bfloat16 K[kC * kS128];
  __nv_bfloat16 Q[kC * kS128];
  __nv_bfloat16 V[kC * kS128];
  float G[kC * kG];                 // g, then gamma (running sum over the chunk), per channel
  __nv_bfloat16 KB[kC * kS128];     // K o e^(gamma - gamma_r) (row block reference); later K o e^gamma
  __nv_bfloat16 QB[kC * kS128];     // Q o e^(gamma - gamma_r)
  __nv_bfloat16 KI[160 * kS128];    // per row block I: K_j o e^(gamma_rI - gamma_j), j < 16 (I + 1)
  float A[kC * kSF];
  float X[kC * kS4];
  alignas(16) float R[3 * 256];
  __nv_bfloat16 T2[kC * kS64];      // X diag(beta)
  float bet[kC];
  float tot[4 * kD];               // scratch of the channel running sums
};
static_assert(sizeof(KdaPrepSmem) <= 227 * 1024, "fits one SM");

// dst[c] = src[c] e^(a[c] - b[c]) (rounded to bf16) for the eight channels
// c of {4q, .., 4q + 3} and {64 + 4q, .., 64 + 4q + 3} of one 128-channel row:
// sixteen lanes with q = 0 .. 15 read and write contiguous runs, which keeps
// the shared-memory accesses free of bank conflicts.
__device__ __forceinline__ void scale_row8(__nv_bfloat16* dst, const __nv_bfloat16* src, const float* a,
                                          const float* b, int q) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int c = 64 * half + 4 * q;
    const float4 av = *reinterpret_cast<const float4*>(a + c), bv = *reinterpret_cast<const float4*>(b + c);
    const uint2 x = *reinterpret_cast<const uint2*>(src + c);
    const float2 x0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
    const float2 x1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
    *reinterpret_cast<uint2*>(dst + c) =
        make_uint2(pack2(x0.x * __expf(av.x - bv.x), x0.y * __expf(av.y - bv.y)),
                   pack2(x1.x * __expf(av.z - bv.z), x1.y * __expf(av.w - bv.w)));
  }
}

// f[u] = e^(a[u] - b[u]) for eight consecutive channels (16-byte aligned rows).
__device__ __forceinline__ void scaled_factors(float (&f)[8], const float* a, const float* b) {
  const float4 a0 = *reinterpret_cast<const float4*>(a), a1 = *reinterpret_cast<const float4*>(a + 4);
  const float4 b0 = *reinterpret_cast<const float4*>(b), b1 = *reinterpret_cast<const float4*>(b + 4);
  f[0] = __expf(a0.x - b0.x), f[1] = __expf(a0.y - b0.y), f[2] = __expf(a0.z - b0.z), f[3] = __expf(a0.w - b0.w);
  f[4] = __expf(a1.x - b1.x), f[5] = __expf(a1.y - b1.y), f[6] = __expf(a1.z - b1.z), f[7] = __expf(a1.w - b1.w);
}
// Eight bf16 values times f, rounded back to bf16.
__device__ __forceinline__ uint4 scale8(const uint4 x, const float (&f)[8]) {
  const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&x);
  uint32_t o[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 t = __bfloat1622float2(v[u]);
    o[u] = pack2(t.x * f[2 * u], t.y * f[2 * u + 1]);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Row offset of block I's scaled K copy inside KI (blocks of 16, 32, 48, 64 rows).
__device__ __forceinline__ int ki_row0(int I) { return 8 * I * (I + 1); }

// kBwd (the backward's recomputation) also stores X and the unscaled A.
template <bool kBwd>
__global__ void __launch_bounds__(kLocalThreads) kda_prep_kernel(GdnParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  KdaPrepSmem& sm = *reinterpret_cast<KdaPrepSmem*>(smem_raw);
  constexpr int nt = kLocalThreads;
  grid_dependency_wait();
  const int c = blockIdx.x, h = blockIdx.y;
  const int n_chunks = __ldcg(p.hdr);
  const int4 ch = p.chunks[c];
  if (c >= n_chunks) return;
  const int len = chunk_len(ch, p.total);
  if (len <= 0) return;  // only with a boundary list that breaks its rules
  const int t0 = ch.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sK = smem_u32(sm.K), sQ = smem_u32(sm.Q), sV = smem_u32(sm.V), sKB = smem_u32(sm.KB),
                 sQB = smem_u32(sm.QB), sKI = smem_u32(sm.KI);
  // two copy groups: K, Q and the gates first; V (needed only for U) second
  load_rows128(sK, p.k, t0, len, h, p.nh, tid, nt);
  load_rows128(sQ, p.q, t0, len, h, p.nh, tid, nt);
  for (int e = tid; e < kC * 32; e += nt) {  // g rows, 32 pieces of 16 bytes each
    const int r = e >> 5, cc = (e & 31) * 4;
    const bool ok = r < len;
    cp_async16(smem_u32(&sm.G[r * kG + cc]), p.g + ((size_t)(t0 + (ok ? r : 0)) * p.nh + h) * kD + cc, ok);
  }
  cp_async_commit();
  load_rows128(sV, p.v, t0, len, h, p.nh, tid, nt);
  cp_async_commit();
  if (tid < kC) sm.bet[tid] = tid < len ? p.beta[(size_t)(t0 + tid) * p.nh + h] : 0.f;
  cp_async_wait<1>();
  __syncthreads();
  // gamma per channel (rows past the chunk add zeros).  Every log decay must
  // be above kKdaMinLogDecay (the block-referenced products need the decay of
  // 15 tokens within float range); anything else, NaN included, is reported
  // in the status word.
  if (chan_running_sum<true>(sm.G, sm.tot, tid) && tid == 0 && p.status) atomicExch(p.status, kStatusGateRange);
  // scaled operands: KB, QB (reference = the row's block start) and the KI
  // copies, eight channels per thread (16-byte loads and stores)
  for (int e = tid; e < kC * kD / 8; e += nt) {
    const int i = e >> 4, q = e & 15;
    const int r = i & ~15;
    scale_row8(&sm.KB[i * kS128], &sm.K[i * kS128], &sm.G[i * kG], &sm.G[r * kG], q);
    scale_row8(&sm.QB[i * kS128], &sm.Q[i * kS128], &sm.G[i * kG], &sm.G[r * kG], q);
  }
  for (int e = tid; e < 160 * kD / 8; e += nt) {
    const int row = e >> 4, q = e & 15;
    const int I = row < 16 ? 0 : (row < 48 ? 1 : (row < 96 ? 2 : 3));
    const int j = row - ki_row0(I), r = 16 * I;
    scale_row8(&sm.KI[row * kS128], &sm.K[j * kS128], &sm.G[r * kG], &sm.G[j * kG], q);
  }
  __syncthreads();
  // ---- the 10 blocks (I, J <= I) of 16 x 16: A and Aqk; warp w < 10 takes block w
  __nv_bfloat16* aqk = p.Aqk + ((size_t)c * p.nh + h) * (kC * kC);
  for (int bl = warp; bl < 10; bl += nt / 32) {
    const int I = bl < 1 ? 0 : (bl < 3 ? 1 : (bl < 6 ? 2 : 3));
    const int J = bl - I * (I + 1) / 2;
    float sa[2][4], sq[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) sa[n][e] = sq[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t ak[4], aq[4], b[4];
      ldsm_x4(ak, frag_a(sKB, kS128, 16 * I, 16 * kk, lane));
      ldsm_x4(aq, frag_a(sQB, kS128, 16 * I, 16 * kk, lane));
      ldsm_x4(b, frag_bt(sKI, kS128, ki_row0(I) + 16 * J, 16 * kk, lane));
      mma_bf16(sa[0], ak, b[0], b[1]);
      mma_bf16(sa[1], ak, b[2], b[3]);
      mma_bf16(sq[0], aq, b[0], b[1]);
      mma_bf16(sq[1], aq, b[2], b[3]);
    }
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = 16 * I + (lane >> 2) + 8 * hr;
        const int j = 16 * J + 8 * n + 2 * (lane & 3);
        const float bi = sm.bet[i];
        sm.A[i * kSF + j] = j < i ? bi * sa[n][2 * hr] : 0.f;
        sm.A[i * kSF + j + 1] = j + 1 < i ? bi * sa[n][2 * hr + 1] : 0.f;
        if (kBwd) {
          float* ar = p.Araw + ((size_t)c * p.nh + h) * (kC * kC) + i * kC + j;
          *reinterpret_cast<float2*>(ar) = make_float2(j < i ? sa[n][2 * hr] : 0.f, j + 1 < i ? sa[n][2 * hr + 1] : 0.f);
        }
        *reinterpret_cast<uint32_t*>(aqk + i * kC + j) =
            pack2(j <= i ? sq[n][2 * hr] : 0.f, j + 1 <= i ? sq[n][2 * hr + 1] : 0.f);
      }
  }
  // blocks above the diagonal: zero
  for (int e = tid; e < 6 * 256; e += nt) {
    const int blk = e >> 8, r = (e >> 4) & 15, cc = e & 15;
    const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
    const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
    const int i = 16 * bi + r, j = 16 * bj + cc;
    sm.A[i * kSF + j] = 0.f;
    aqk[i * kC + j] = __float2bfloat16_rn(0.f);
    if (kBwd) p.Araw[((size_t)c * p.nh + h) * (kC * kC) + i * kC + j] = 0.f;
  }
  __syncthreads();
  wy_inverse<kS4, kLocalThreads>(sm.A, sm.X, sm.R, tid);
  if (kBwd) {
    float* xw = p.Xw + ((size_t)c * p.nh + h) * (kC * kC);
    for (int e = tid; e < kC * kC; e += nt) xw[e] = sm.X[(e >> 6) * kS4 + (e & 63)];
  }
  // ---- T2 = X diag(beta); KB <- K o e^gamma; QB, KC, e^gamma_last to the workspace
  for (int e = tid; e < kC * kC / 2; e += nt) {
    const int i = e >> 5, j = (e & 31) * 2;
    *reinterpret_cast<uint32_t*>(&sm.T2[i * kS64 + j]) =
        pack2(sm.X[i * kS4 + j] * sm.bet[j], sm.X[i * kS4 + j + 1] * sm.bet[j + 1]);
  }
  const int last = len - 1;
  for (int e = tid; e < kC * kD / 8; e += nt) {
    const int i = e >> 4, cc = (e & 15) * 8;
    float eg[8], ec[8];
    const float4 g0 = *reinterpret_cast<const float4*>(&sm.G[i * kG + cc]);
    const float4 g1 = *reinterpret_cast<const float4*>(&sm.G[i * kG + cc + 4]);
    eg[0] = __expf(g0.x), eg[1] = __expf(g0.y), eg[2] = __expf(g0.z), eg[3] = __expf(g0.w);
    eg[4] = __expf(g1.x), eg[5] = __expf(g1.y), eg[6] = __expf(g1.z), eg[7] = __expf(g1.w);
    scaled_factors(ec, &sm.G[last * kG + cc], &sm.G[i * kG + cc]);
    const uint4 kv = *reinterpret_cast<const uint4*>(&sm.K[i * kS128 + cc]);
    *reinterpret_cast<uint4*>(&sm.KB[i * kS128 + cc]) = scale8(kv, eg);
    if (i < len) {
      const size_t off = ((size_t)(t0 + i) * p.nh + h) * kD + cc;
      *reinterpret_cast<uint4*>(p.QB + off) = scale8(*reinterpret_cast<const uint4*>(&sm.Q[i * kS128 + cc]), eg);
      *reinterpret_cast<uint4*>(p.KC + off) = scale8(kv, ec);
    }
  }
  if (tid < kD) p.Bc[((size_t)c * p.nh + h) * kD + tid] = __expf(sm.G[last * kG + tid]);
  cp_async_wait<0>();  // V
  __syncthreads();
  // ---- W = T2 (K o e^gamma), U = T2 V: warp w rows [16 (w % 4), +16) x columns [32 (w / 4), +32)
  const int r0 = 16 * (warp & 3), d0 = 32 * (warp >> 2);
  float cw[4][4], cu[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) cw[n][e] = cu[n][e] = 0.f;
  const uint32_t sT2 = smem_u32(sm.T2);
#pragma unroll
  for (int kk = 0; kk < kC / 16; ++kk) {
    uint32_t a[4];
    ldsm_x4(a, frag_a(sT2, kS64, r0, 16 * kk, lane));
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t bk[4], bv[4];
      ldsm_x4_t(bk, frag_b(sKB, kS128, 16 * kk, d0 + 16 * np, lane));
      ldsm_x4_t(bv, frag_b(sV, kS128, 16 * kk, d0 + 16 * np, lane));
      mma_bf16(cw[2 * np], a, bk[0], bk[1]);
      mma_bf16(cw[2 * np + 1], a, bk[2], bk[3]);
      mma_bf16(cu[2 * np], a, bv[0], bv[1]);
      mma_bf16(cu[2 * np + 1], a, bv[2], bv[3]);
    }
  }
  __syncthreads();  // K, V no longer read: stage W in K's place, U in V's
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = r0 + (lane >> 2) + 8 * hr;
      const int j = d0 + 8 * n + 2 * (lane & 3);
      *reinterpret_cast<uint32_t*>(&sm.K[i * kS128 + j]) = pack2(cw[n][2 * hr], cw[n][2 * hr + 1]);
      *reinterpret_cast<uint32_t*>(&sm.V[i * kS128 + j]) = pack2(cu[n][2 * hr], cu[n][2 * hr + 1]);
    }
  __syncthreads();
  for (int e = tid; e < kC * 16; e += nt) {
    const int r = e >> 4, cc = (e & 15) * 8;
    if (r < len) {
      const size_t off = ((size_t)(t0 + r) * p.nh + h) * kD + cc;
      *reinterpret_cast<uint4*>(p.W + off) = *reinterpret_cast<const uint4*>(&sm.K[r * kS128 + cc]);
      *reinterpret_cast<uint4*>(p.U + off) = *reinterpret_cast<const uint4*>(&sm.V[r * kS128 + cc]);
    }
  }
}

// ============================================================== state + output
// The state passes run as a pipeline of three stages.  A producer warp fills
// stage c % 3 with the pass's chunk c: the chunk's three 64 x 128 token-row
// tiles (W, K, Q) and its 64 x 64 Aq block, swizzled by 128 bytes (see
// sw128), and the CTA's 32 value columns of U (forward) or dO (backward),
// swizzled by 64 bytes (see sw64), all by TMA on the stage's full barrier;
// the gates by plain loads.  The eight compute warps release the stage on
// its empty barrier when they are done with it.  So the compute warps spend
// nothing on loads, and need no barrier at the end of a step.
// Rows past the end of the tensor arrive as zeros; rows past the chunk's end
// that belong to the next segment are zeroed once the tiles have landed, so
// no chunk reads another segment.
constexpr int kTileBytes = kC * kD * 2;  // 64 x 128 bf16: two 8 KB halves
constexpr int kColsBytes = kC * kDvb * 2;  // 64 x 32 bf16
constexpr uint32_t kStageTxBytes = 3 * kTileBytes + kC * kC * 2 + kColsBytes;
constexpr int kStateBlock = kStateThreads + 32;  // eight compute warps and the producer

// The TMA maps of the state passes.  W, K and Q ([T, H, 128] bf16; Kimi Delta
// reads K o e^(gamma_last - gamma) and Q o e^gamma) as 4-D tensors (64
// columns, token, column half, head), box 64 x 64 tokens x 2 halves x 1 head:
// one copy lands a whole 64 x 128 tile as its two swizzled halves.  Aqk
// ([chunks x H, 64, 64] bf16), box one block.  U and dO ([T, H, 128] bf16),
// box 32 columns x 1 head x 64 tokens.
struct StateMaps {
  CUtensorMap w, k, q, aq, u, d_o;
};

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

struct alignas(1024) StateStage {
  __nv_bfloat16 W[kC * kD];      // swizzled; W, K, Q are consecutive
  __nv_bfloat16 K[kC * kD];      // swizzled
  __nv_bfloat16 Q[kC * kD];      // swizzled
  __nv_bfloat16 Aq[kC * kC];     // swizzled
  __nv_bfloat16 cols[kC * kDvb]; // 64-byte swizzle: value columns of U (forward) or dO (backward)
  float gam[kD];  // gamma of the chunk's tokens; with a decay per channel, e^gamma_last per channel
};
static_assert(offsetof(StateStage, K) == kTileBytes && offsetof(StateStage, Q) == 2 * kTileBytes &&
                  offsetof(StateStage, Aq) == 3 * kTileBytes && offsetof(StateStage, cols) % 1024 == 0,
              "TMA tiles at 1024-byte offsets");
constexpr int kStateStages = 3;
struct StatePipe {
  StateStage st[kStateStages];
  uint64_t full[kStateStages];   // the producer's copies of stage s have landed
  uint64_t empty[kStateStages];  // the eight compute warps are done with stage s
  int abort;                     // a wait of this CTA gave up
};
struct StateSmem {
  StatePipe pp;
  __nv_bfloat16 H[kD * kS32];   // the state at the chunk start, bf16 (B operand)
  __nv_bfloat16 E[kC * kS32];   // E (bf16)
  __nv_bfloat16 E2[kC * kS32];  // diag(e^(gamma_last - gamma)) E (bf16)
};
// The launch adds 1024 bytes of slack to align the stages.
static_assert(sizeof(StateSmem) + 1024 <= 227 * 1024, "the state CTA's shared memory fits one SM");

__device__ __forceinline__ uint8_t* align1024(uint8_t* raw) {
  return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

// Byte offset of element (r, c) of the 64 x 32 value columns, 64-byte rows
// with the 64-byte swizzle (16-byte chunk j of row r at chunk j ^ (r / 2 % 4)).
// Eight consecutive rows of one chunk fall in eight different bank groups.
__device__ __forceinline__ uint32_t sw64(int r, int c) {
  return (uint32_t)(r * 64 + (((((c >> 3) ^ (r >> 1)) & 3)) << 4) + (c & 7) * 2);
}
__device__ __forceinline__ float2 cols_pair(const StateStage& s, int r, int c) {
  return __bfloat1622float2(
      *reinterpret_cast<const __nv_bfloat162*>(reinterpret_cast<const uint8_t*>(s.cols) + sw64(r, c)));
}
// frag_b over the value columns.
__device__ __forceinline__ uint32_t frag_b_cols(uint32_t base, int k0, int n0, int lane) {
  return base + sw64(k0 + (lane & 15), n0 + ((lane >> 4) << 3));
}

// The 256 compute threads' own barrier (the producer warp never joins it).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool compute_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, 1, 256, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Rows [len, 64) of the stage's token-row tiles and value columns to zero
// (each keeps row r in one run of bytes, whatever the swizzle).
__device__ __forceinline__ void zero_tail_rows(StateStage& s, int len, int tid) {
  uint8_t* base = reinterpret_cast<uint8_t*>(s.W);
  const int n = (kC - len) * 8;  // 16-byte chunks per half tile
  for (int e = tid; e < 6 * n; e += kStateThreads) {
    const int hf = e / n, x = e - hf * n;
    *reinterpret_cast<uint4*>(base + hf * (kTileBytes / 2) + len * 128 + x * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  uint8_t* cols = reinterpret_cast<uint8_t*>(s.cols);
  for (int e = tid; e < (kC - len) * 4; e += kStateThreads)
    *reinterpret_cast<uint4*>(cols + len * 64 + e * 16) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();  // before the stage's next TMA overwrite
}

// Lane 0 after a wait gave up: waits (bounded again) for the copies of the
// pass's chunks [c0, c1) that may still be in flight, so that the CTA leaves
// no copy writing its shared memory.
__device__ __forceinline__ void drain_copies(const uint64_t* full, int c0, int c1) {
  for (int c = c0; c < c1; ++c) {
    const uint32_t bar = smem_u32(&full[c % kStateStages]);
    const uint32_t parity = (uint32_t)(c / kStateStages) & 1u;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity) && global_timer_ns() - t0 < VSW_WAIT_TIMEOUT_NS) {
    }
  }
}

// The producer warp.  The pass visits the segment's chunks in order
// (forward) or in reverse (backward); its chunk c goes to stage c % 3 once
// the compute warps have released the stage's previous chunk c - 3.
template <bool kChan, bool kReverse>
__device__ __forceinline__ void state_producer(StatePipe& pp, const StateMaps& m, const GdnParams& p, const int4& sg,
                                               int nch, int h, int vb, int lane) {
  const CUtensorMap* cols_map = kReverse ? &m.d_o : &m.u;
  for (int c = 0; c < nch; ++c) {
    const int st = c % kStateStages;
    if (c >= kStateStages &&
        !mbar_wait_warp(smem_u32(&pp.empty[st]), (uint32_t)(c / kStateStages - 1) & 1u, &pp.abort, p.status)) {
      if (lane == 0) drain_copies(pp.full, c - kStateStages, c);
      return;
    }
    const int ci = kReverse ? nch - 1 - c : c;
    const int chunk = sg.x + ci;
    const int4 ch = seg_chunk(sg, ci);
    const int len = chunk_len(ch, p.total), t0 = len > 0 ? ch.x : 0;
    StateStage& s = pp.st[st];
    if (kChan) {
      *reinterpret_cast<float4*>(&s.gam[4 * lane]) =
          *reinterpret_cast<const float4*>(p.Bc + ((size_t)chunk * p.nh + h) * kD + 4 * lane);
    } else {
      for (int i = lane; i < kC; i += 32) s.gam[i] = i < len ? p.gam[(size_t)h * p.total + t0 + i] : 0.f;
    }
    __syncwarp();
    if (lane == 0) {
      const uint32_t bar = smem_u32(&pp.full[st]);
      // generic-proxy accesses of the stage's last use before the async-proxy overwrite
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, kStageTxBytes);  // also publishes the gates
      tma_load_4d(smem_u32(s.W), &m.w, bar, 0, t0, 0, h);
      tma_load_4d(smem_u32(s.K), &m.k, bar, 0, t0, 0, h);
      tma_load_4d(smem_u32(s.Q), &m.q, bar, 0, t0, 0, h);
      tma_load_3d(smem_u32(s.Aq), &m.aq, bar, 0, 0, chunk * p.nh + h);
      tma_load_3d(smem_u32(s.cols), cols_map, bar, kDvb * vb, h, t0);
    }
  }
}

// Pipeline set-up of a state CTA: barriers, then (for the producer warp) the
// whole production.  Returns true for the compute threads.
template <bool kChan, bool kReverse>
__device__ __forceinline__ bool state_pipe_start(StatePipe& pp, const StateMaps& m, const GdnParams& p,
                                                 const int4& sg, int nch, int h, int vb, int tid) {
  if (tid == 0) {
    for (int i = 0; i < kStateStages; ++i) {
      mbar_init(smem_u32(&pp.full[i]), 1);
      mbar_init(smem_u32(&pp.empty[i]), kStateThreads / 32);
    }
    pp.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (tid >= kStateThreads) {
    state_producer<kChan, kReverse>(pp, m, p, sg, nch, h, vb, tid & 31);
    return false;
  }
  return true;
}

// A compute warp is done with stage st.
__device__ __forceinline__ void release_stage(StatePipe& pp, int st, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&pp.empty[st]));
}

// Eight compute warps.  Warp w computes, of the chunk's 64 x 32 products (E,
// Q H, O), rows [16 (w % 4), +16) x columns [16 (w / 4), +16), and holds rows
// [16 w, +16) of the 128 x 32 state.
// kOut: O goes to p.o.  kStore (for the backward): the bf16 state at every
// chunk start and every chunk's E go to the workspace.  The backward's own
// recomputation stores without O; a saving forward does both.
// kChan (Kimi Delta): K and Q arrive pre-scaled (KC, QB), so E and O take no
// per-token factor, and the state decays by e^gamma_last per channel (row).
template <bool kOut, bool kStore, bool kChan>
__global__ void __launch_bounds__(kStateBlock) gdn_state_kernel(const __grid_constant__ StateMaps maps,
                                                                GdnParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  StateSmem& sm = *reinterpret_cast<StateSmem*>(align1024(smem_raw));
  grid_dependency_wait();
  const int per_seg = p.nh * (kD / kDvb);
  const int r = blockIdx.x / per_seg, rem = blockIdx.x - r * per_seg;
  const int h = rem / (kD / kDvb), vb = rem - h * (kD / kDvb);
  if (r >= p.hdr[1]) return;
  const int4 sg = p.segs[r];
  // (the chunk count clamped to the table: the saved backward reads a
  // workspace that only its caller vouches for)
  const int first = sg.x, nch = min(sg.y, min(p.hdr[0], p.max_chunks) - sg.x);
  if (first < 0 || nch <= 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (!state_pipe_start<kChan, false>(sm.pp, maps, p, sg, nch, h, vb, tid)) return;
  const int r0 = 16 * (warp & 3);   // token rows of the E / O products
  const int n0 = 16 * (warp >> 2);  // their value columns
  const int m0 = 16 * warp;         // state rows (d_k)
  float hreg[4][4];                 // state rows [m0, +16) x 32 columns, as mma accumulators (n-tile n)
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) hreg[n][e] = 0.f;
  const uint32_t sH = smem_u32(sm.H), sE = smem_u32(sm.E), sE2 = smem_u32(sm.E2);
  for (int ci = 0; ci < nch; ++ci) {
    const int st = ci % kStateStages;
    StateStage& s = sm.pp.st[st];
    const int4 ch = seg_chunk(sg, ci);
    const int t0 = ch.x, len = chunk_len(ch, p.total);
    const bool landed =
        mbar_wait(smem_u32(&sm.pp.full[st]), (uint32_t)(ci / kStateStages) & 1u, &sm.pp.abort, p.status);
    if (landed && len > 0 && len < kC) zero_tail_rows(s, len, tid);
    // H (bf16) for this chunk's products.  Its last readers (the previous
    // chunk's E / Q H products) finished before that chunk's second barrier.
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = m0 + (lane >> 2) + 8 * hr;
        const int j = 8 * n + 2 * (lane & 3);
        *reinterpret_cast<uint32_t*>(&sm.H[i * kS32 + j]) = pack2(hreg[n][2 * hr], hreg[n][2 * hr + 1]);
      }
    if (compute_sync_or(!landed)) return;  // the producer drains the copies in flight
    if (kStore) {
      // H (bf16) of this chunk start: 128 rows x 64 bytes of this CTA's columns
      __nv_bfloat16* dst = p.H0 + ((size_t)(first + ci) * p.nh + h) * (kD * kD) + kDvb * vb;
      for (int e = tid; e < kD * 4; e += kStateThreads) {
        const int rr = e >> 2, cc = (e & 3) * 8;
        *reinterpret_cast<uint4*>(dst + rr * kD + cc) = *reinterpret_cast<const uint4*>(&sm.H[rr * kS32 + cc]);
      }
    }
    if (len <= 0) {  // only with a boundary list that breaks its rules
      compute_sync();  // the H reads above before the next chunk's H write
      release_stage(sm.pp, st, lane);
      continue;
    }
    const uint32_t sW = smem_u32(s.W), sK = smem_u32(s.K), sQ = smem_u32(s.Q), sAq = smem_u32(s.Aq);
    const float g_last = kChan ? 0.f : s.gam[len - 1];
    // ---- E = U - W H and Q H
    float ce[2][4], cq[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) ce[n][e] = cq[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t aw[4], aq[4], b[4];
      ldsm_x4(aw, frag_a_sw(sW, r0, 16 * kk, lane));
      ldsm_x4(aq, frag_a_sw(sQ, r0, 16 * kk, lane));
      ldsm_x4_t(b, frag_b(sH, kS32, 16 * kk, n0, lane));
      mma_bf16(ce[0], aw, b[0], b[1]);
      mma_bf16(ce[1], aw, b[2], b[3]);
      if (kOut) {
        mma_bf16(cq[0], aq, b[0], b[1]);
        mma_bf16(cq[1], aq, b[2], b[3]);
      }
    }
    // E and E2 overwrite the previous chunk's, whose readers (its O and state
    // update) finished before this chunk's first barrier.
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = r0 + (lane >> 2) + 8 * hr;
        const int j = n0 + 8 * n + 2 * (lane & 3);
        const float2 u = cols_pair(s, i, j);
        const float e0 = u.x - ce[n][2 * hr], e1 = u.y - ce[n][2 * hr + 1];
        const float w = i < len ? (kChan ? 1.f : __expf(g_last - s.gam[i])) : 0.f;
        *reinterpret_cast<uint32_t*>(&sm.E[i * kS32 + j]) = pack2(e0, e1);
        *reinterpret_cast<uint32_t*>(&sm.E2[i * kS32 + j]) = pack2(e0 * w, e1 * w);
      }
    compute_sync();
    if (kStore) {
      for (int e = tid; e < kC * 4; e += kStateThreads) {
        const int rr = e >> 2, cc = (e & 3) * 8;
        if (rr < len)
          *reinterpret_cast<uint4*>(p.E + ((size_t)(t0 + rr) * p.nh + h) * kD + kDvb * vb + cc) =
              *reinterpret_cast<const uint4*>(&sm.E[rr * kS32 + cc]);
      }
    }
    if (kOut) {
      // ---- O = scale (e^gamma Q H + Aq E)
      float co[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) co[n][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < kC / 16; ++kk) {
        uint32_t a[4], b[4];
        ldsm_x4(a, frag_a_sw(sAq, r0, 16 * kk, lane));
        ldsm_x4_t(b, frag_b(sE, kS32, 16 * kk, n0, lane));
        mma_bf16(co[0], a, b[0], b[1]);
        mma_bf16(co[1], a, b[2], b[3]);
      }
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = r0 + (lane >> 2) + 8 * hr;
        if (i < len) {
          const float eg = kChan ? 1.f : __expf(s.gam[i]);
          __nv_bfloat16* orow = p.o + ((size_t)(t0 + i) * p.nh + h) * kD + kDvb * vb + n0;
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            const int j = 8 * n + 2 * (lane & 3);
            *reinterpret_cast<uint32_t*>(orow + j) = pack2(p.scale * (eg * cq[n][2 * hr] + co[n][2 * hr]),
                                                           p.scale * (eg * cq[n][2 * hr + 1] + co[n][2 * hr + 1]));
          }
        }
      }
    }
    // ---- H = e^gamma_last H + K^T E2 (state rows [m0, +16); K^T read from K[token][d_k])
    // rows m0 + lane / 4 (elements 0, 1) and + 8 (elements 2, 3)
    const float dl0 = kChan ? s.gam[m0 + (lane >> 2)] : __expf(g_last);
    const float dl1 = kChan ? s.gam[m0 + (lane >> 2) + 8] : dl0;
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      hreg[n][0] *= dl0;
      hreg[n][1] *= dl0;
      hreg[n][2] *= dl1;
      hreg[n][3] *= dl1;
    }
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) {
      uint32_t a[4], b0[4], b1[4];
      ldsm_x4_t(a, frag_bt_sw(sK, 16 * kk, m0, lane));
      ldsm_x4_t(b0, frag_b(sE2, kS32, 16 * kk, 0, lane));
      ldsm_x4_t(b1, frag_b(sE2, kS32, 16 * kk, 16, lane));
      mma_bf16(hreg[0], a, b0[0], b0[1]);
      mma_bf16(hreg[1], a, b0[2], b0[3]);
      mma_bf16(hreg[2], a, b1[0], b1[1]);
      mma_bf16(hreg[3], a, b1[2], b1[3]);
    }
    release_stage(sm.pp, st, lane);
  }
}


// ============================================================== backward: state gradient
// Reverse over a segment's chunks, per (segment, head, 32 value columns),
// carrying dH = dL/dH1 (the state at the chunk end; zero after the last
// chunk) in registers:
//     dE  = scale Aq^T dO + diag(e^(gamma_last - gamma)) K dH
//     dH0 = e^gamma_last dH + scale Q^T diag(e^gamma) dO - W^T dE
// dE and the bf16 dH of every chunk go to the workspace for the local pass.
// The same pipeline as the forward state pass, over the chunks in reverse.
struct BwdStateSmem {
  StatePipe pp;                  // W, K, Q, Aq, dO, gates
  __nv_bfloat16 H[kD * kS32];    // dH (bf16)
  __nv_bfloat16 E[kC * kS32];    // dE (bf16)
  __nv_bfloat16 G[kC * kS32];    // scale e^gamma dO (bf16)
};
static_assert(sizeof(BwdStateSmem) + 1024 <= 227 * 1024, "the backward state CTA's shared memory fits one SM");

// kChan (Kimi Delta): KC and QB replace K and Q (no per-token factors), and
// the gradient decays by e^gamma_last per channel (row).
template <bool kChan>
__global__ void __launch_bounds__(kStateBlock) gdn_bwd_state_kernel(const __grid_constant__ StateMaps maps,
                                                                    GdnParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  BwdStateSmem& sm = *reinterpret_cast<BwdStateSmem*>(align1024(smem_raw));
  grid_dependency_wait();
  const int per_seg = p.nh * (kD / kDvb);
  const int r = blockIdx.x / per_seg, rem = blockIdx.x - r * per_seg;
  const int h = rem / (kD / kDvb), vb = rem - h * (kD / kDvb);
  if (r >= p.hdr[1]) return;
  const int4 sg = p.segs[r];
  // (the chunk count clamped to the table: the saved backward reads a
  // workspace that only its caller vouches for)
  const int first = sg.x, nch = min(sg.y, min(p.hdr[0], p.max_chunks) - sg.x);
  if (first < 0 || nch <= 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (!state_pipe_start<kChan, true>(sm.pp, maps, p, sg, nch, h, vb, tid)) return;
  const int r0 = 16 * (warp & 3);   // token rows of dE
  const int n0 = 16 * (warp >> 2);  // its value columns
  const int m0 = 16 * warp;         // dH rows (d_k)
  float dh[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) dh[n][e] = 0.f;
  const uint32_t sH = smem_u32(sm.H), sE = smem_u32(sm.E), sG = smem_u32(sm.G);
  // step ci (0 = the segment's last chunk) is chunk first + nch - 1 - ci, in stage ci % 3
  for (int ci = 0; ci < nch; ++ci) {
    const int st = ci % kStateStages;
    const int chunk = first + nch - 1 - ci;
    StateStage& s = sm.pp.st[st];
    const int4 ch = seg_chunk(sg, nch - 1 - ci);
    const int t0 = ch.x, len = chunk_len(ch, p.total);
    const bool landed =
        mbar_wait(smem_u32(&sm.pp.full[st]), (uint32_t)(ci / kStateStages) & 1u, &sm.pp.abort, p.status);
    if (landed && len > 0 && len < kC) zero_tail_rows(s, len, tid);
    // dH (bf16); its last readers (the previous step's dE products and dH1
    // store) finished before that step's second barrier
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = m0 + (lane >> 2) + 8 * hr;
        const int j = 8 * n + 2 * (lane & 3);
        *reinterpret_cast<uint32_t*>(&sm.H[i * kS32 + j]) = pack2(dh[n][2 * hr], dh[n][2 * hr + 1]);
      }
    if (compute_sync_or(!landed)) return;  // the producer drains the copies in flight
    {
      __nv_bfloat16* dst = p.dH1 + ((size_t)chunk * p.nh + h) * (kD * kD) + kDvb * vb;
      for (int e = tid; e < kD * 4; e += kStateThreads) {
        const int rr = e >> 2, cc = (e & 3) * 8;
        *reinterpret_cast<uint4*>(dst + rr * kD + cc) = *reinterpret_cast<const uint4*>(&sm.H[rr * kS32 + cc]);
      }
    }
    if (len <= 0) {  // only with a boundary list that breaks its rules
      compute_sync();  // the dH reads above before the next step's dH write
      release_stage(sm.pp, st, lane);
      continue;
    }
    const uint32_t sK = smem_u32(s.K), sQ = smem_u32(s.Q), sW = smem_u32(s.W), sAq = smem_u32(s.Aq),
                   sdO = smem_u32(s.cols);
    const float g_last = kChan ? 0.f : s.gam[len - 1];
    // ---- dE = scale Aq^T dO + diag(e^(gamma_last - gamma)) K dH
    float ca[2][4], ck[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) ca[n][e] = ck[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) {
      uint32_t a[4], b[4];
      ldsm_x4_t(a, frag_bt_sw(sAq, 16 * kk, r0, lane));  // Aq^T: Aq stored [i][j]
      ldsm_x4_t(b, frag_b_cols(sdO, 16 * kk, n0, lane));
      mma_bf16(ca[0], a, b[0], b[1]);
      mma_bf16(ca[1], a, b[2], b[3]);
    }
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t a[4], b[4];
      ldsm_x4(a, frag_a_sw(sK, r0, 16 * kk, lane));
      ldsm_x4_t(b, frag_b(sH, kS32, 16 * kk, n0, lane));
      mma_bf16(ck[0], a, b[0], b[1]);
      mma_bf16(ck[1], a, b[2], b[3]);
    }
    // dE and G overwrite the previous step's, whose readers finished before
    // this step's first barrier
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = r0 + (lane >> 2) + 8 * hr;
      const float w = i < len ? (kChan ? 1.f : __expf(g_last - s.gam[i])) : 0.f;
      const float m = i < len ? p.scale : 0.f;
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const int j = n0 + 8 * n + 2 * (lane & 3);
        *reinterpret_cast<uint32_t*>(&sm.E[i * kS32 + j]) =
            pack2(m * ca[n][2 * hr] + w * ck[n][2 * hr], m * ca[n][2 * hr + 1] + w * ck[n][2 * hr + 1]);
      }
    }
    // scale e^gamma dO, the B operand of Q^T (.) below
    for (int e = tid; e < kC * 16; e += kStateThreads) {
      const int i = e >> 4, j = (e & 15) * 2;
      const float m = i < len ? p.scale * (kChan ? 1.f : __expf(s.gam[i])) : 0.f;
      const float2 d = cols_pair(s, i, j);
      *reinterpret_cast<uint32_t*>(&sm.G[i * kS32 + j]) = pack2(m * d.x, m * d.y);
    }
    compute_sync();
    for (int e = tid; e < kC * 4; e += kStateThreads) {
      const int rr = e >> 2, cc = (e & 3) * 8;
      if (rr < len)
        *reinterpret_cast<uint4*>(p.dE + ((size_t)(t0 + rr) * p.nh + h) * kD + kDvb * vb + cc) =
            *reinterpret_cast<const uint4*>(&sm.E[rr * kS32 + cc]);
    }
    // ---- dH = e^gamma_last dH + Q^T G - W^T dE (rows [m0, +16))
    const float dl0 = kChan ? s.gam[m0 + (lane >> 2)] : __expf(g_last);
    const float dl1 = kChan ? s.gam[m0 + (lane >> 2) + 8] : dl0;
    float cw[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      dh[n][0] *= dl0;
      dh[n][1] *= dl0;
      dh[n][2] *= dl1;
      dh[n][3] *= dl1;
#pragma unroll
      for (int e = 0; e < 4; ++e) cw[n][e] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) {
      uint32_t aq[4], aw[4], g0[4], g1[4], e0[4], e1[4];
      ldsm_x4_t(aq, frag_bt_sw(sQ, 16 * kk, m0, lane));
      ldsm_x4_t(aw, frag_bt_sw(sW, 16 * kk, m0, lane));
      ldsm_x4_t(g0, frag_b(sG, kS32, 16 * kk, 0, lane));
      ldsm_x4_t(g1, frag_b(sG, kS32, 16 * kk, 16, lane));
      ldsm_x4_t(e0, frag_b(sE, kS32, 16 * kk, 0, lane));
      ldsm_x4_t(e1, frag_b(sE, kS32, 16 * kk, 16, lane));
      mma_bf16(dh[0], aq, g0[0], g0[1]);
      mma_bf16(dh[1], aq, g0[2], g0[3]);
      mma_bf16(dh[2], aq, g1[0], g1[1]);
      mma_bf16(dh[3], aq, g1[2], g1[3]);
      mma_bf16(cw[0], aw, e0[0], e0[1]);
      mma_bf16(cw[1], aw, e0[2], e0[3]);
      mma_bf16(cw[2], aw, e1[0], e1[1]);
      mma_bf16(cw[3], aw, e1[2], e1[3]);
    }
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) dh[n][e] -= cw[n][e];
    release_stage(sm.pp, st, lane);
  }
}

// ============================================================== backward: local, with the states
// Per (chunk, head), everything that needs the bf16 state at the chunk start
// (H0) or the gradient at its end (dH1), with dAqk = lower(scale dO E^T) and
// DG = dAqk o Gamma:
//     dq   = scale diag(e^gamma) dO H0^T + DG K                    (final)
//     dW   = -dE H0^T                                              (to the workspace)
//     dKa  = diag(e^(gamma_last - gamma)) E dH1^T + DG^T Q         (to the workspace)
//     dgam = rowsum - colsum of DG o (Q K^T) + scale e^gamma_i <dO_i, (Q H0)_i>
//            - w_i <(K dH1)_i, E_i>, and at the last token + sum_i w_i <(K dH1)_i, E_i>
//            + e^gamma_last <dH1, H0>      (w_i = e^(gamma_last - gamma_i); to the workspace)
struct LocalHSmem {
  __nv_bfloat16 dO[kC * kS128];
  __nv_bfloat16 dE[kC * kS128];
  __nv_bfloat16 E[kC * kS128];
  __nv_bfloat16 Q[kC * kS128];
  __nv_bfloat16 K[kC * kS128];
  __nv_bfloat16 H0[kD * kS128];
  __nv_bfloat16 dH1[kD * kS128];
  __nv_bfloat16 DG[kC * kS64];
  float gam[kC];
  float dgs[kC];
  // Partial sums of dgam, one slot per contributing warp group, added in a
  // fixed order at the end (float atomics would make the bits depend on
  // timing): [0..3] DG o QK row sums, [4..7] minus its column sums, [8..11]
  // the dO . Q H0 and E . K dH1 terms; lw: w_i <(K dH1)_i, E_i> per slot; tw:
  // e^gamma_last <dH1, H0> per warp.
  float part[12][kC];
  float lw[4][kC];
  float tw[kLocalThreads / 32];
  float last;  // the gamma_last terms
};
static_assert(sizeof(LocalHSmem) <= 227 * 1024, "fits one SM");

// Sum over the 4 lanes of a quad (the lanes holding one row of an mma tile).
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

__global__ void __launch_bounds__(kLocalThreads) gdn_bwd_local_h_kernel(GdnParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  LocalHSmem& sm = *reinterpret_cast<LocalHSmem*>(smem_raw);
  constexpr int nt = kLocalThreads;
  grid_dependency_wait();
  const int c = blockIdx.x, h = blockIdx.y;
  // (both loads in flight at once: the table entry is in bounds for every
  // c < max_chunks, and ignored past the number of chunks)
  const int n_chunks = __ldcg(p.hdr);
  const int4 ch = p.chunks[c];
  if (c >= n_chunks) return;
  const int len = chunk_len(ch, p.total);
  if (len <= 0) return;  // only with a boundary list that breaks its rules
  const int t0 = ch.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sdO = smem_u32(sm.dO), sdE = smem_u32(sm.dE), sE = smem_u32(sm.E), sQ = smem_u32(sm.Q),
                 sK = smem_u32(sm.K), sH0 = smem_u32(sm.H0), sdH1 = smem_u32(sm.dH1), sDG = smem_u32(sm.DG);
  // Three copy groups, waited for in the order the products need them:
  // dO, E, Q, K (the masked block DG); H0, dE (dq, dW); dH1 (dKa, dgam).
  load_rows128(sdO, p.dO, t0, len, h, p.nh, tid, nt);
  load_rows128(sE, p.E, t0, len, h, p.nh, tid, nt);
  load_rows128(sQ, p.q, t0, len, h, p.nh, tid, nt);
  load_rows128(sK, p.k, t0, len, h, p.nh, tid, nt);
  cp_async_commit();
  const __nv_bfloat16* h0 = p.H0 + ((size_t)c * p.nh + h) * (kD * kD);
  const __nv_bfloat16* d1 = p.dH1 + ((size_t)c * p.nh + h) * (kD * kD);
  for (int e = tid; e < kD * 16; e += nt) {
    const int r = e >> 4, cc = (e & 15) * 8;
    cp_async16(sH0 + 2u * (uint32_t)(r * kS128 + cc), h0 + r * kD + cc, true);
  }
  load_rows128(sdE, p.dE, t0, len, h, p.nh, tid, nt);
  cp_async_commit();
  for (int e = tid; e < kD * 16; e += nt) {
    const int r = e >> 4, cc = (e & 15) * 8;
    cp_async16(sdH1 + 2u * (uint32_t)(r * kS128 + cc), d1 + r * kD + cc, true);
  }
  cp_async_commit();
  if (tid < kC) {
    sm.gam[tid] = tid < len ? p.gam[(size_t)h * p.total + t0 + tid] : 0.f;
    sm.dgs[tid] = 0.f;
  }
  for (int e = tid; e < 16 * kC; e += nt) (&sm.part[0][0])[e] = 0.f;  // part and lw
  cp_async_wait<2>();
  __syncthreads();
  const float g_last = sm.gam[len - 1];
  const int r0 = 16 * (warp & 3);
  // ---- dO E^T and Q K^T (rows [r0, +16), columns [c0, +16)): DG, and the
  // DG o (Q K^T) row and column sums of dgam.
  {
    const int c0 = 16 * (warp >> 2);
    float s1[2][4], s2[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) s1[n][e] = s2[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t ad[4], aq[4];
      ldsm_x4(ad, frag_a(sdO, kS128, r0, 16 * kk, lane));
      ldsm_x4(aq, frag_a(sQ, kS128, r0, 16 * kk, lane));
#pragma unroll
      for (int np = 0; np < 1; ++np) {
        uint32_t be[4], bk[4];
        ldsm_x4(be, frag_bt(sE, kS128, c0 + 16 * np, 16 * kk, lane));
        ldsm_x4(bk, frag_bt(sK, kS128, c0 + 16 * np, 16 * kk, lane));
        mma_bf16(s1[2 * np], ad, be[0], be[1]);
        mma_bf16(s1[2 * np + 1], ad, be[2], be[3]);
        mma_bf16(s2[2 * np], aq, bk[0], bk[1]);
        mma_bf16(s2[2 * np + 1], aq, bk[2], bk[3]);
      }
    }
    float rsum[2] = {0.f, 0.f};
    float csum[2][2];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      csum[n][0] = csum[n][1] = 0.f;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = r0 + (lane >> 2) + 8 * hr;
        const int j = c0 + 8 * n + 2 * (lane & 3);
        const float gi = sm.gam[i];
        const float d0 = j <= i ? p.scale * s1[n][2 * hr] * __expf(gi - sm.gam[j]) : 0.f;
        const float d1 = j + 1 <= i ? p.scale * s1[n][2 * hr + 1] * __expf(gi - sm.gam[j + 1]) : 0.f;
        *reinterpret_cast<uint32_t*>(&sm.DG[i * kS64 + j]) = pack2(d0, d1);
        const float r_0 = d0 * s2[n][2 * hr], r_1 = d1 * s2[n][2 * hr + 1];
        rsum[hr] += r_0 + r_1;
        csum[n][0] += r_0;
        csum[n][1] += r_1;
      }
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const float x = quad_sum(rsum[hr]);
      if ((lane & 3) == 0) sm.part[warp >> 2][r0 + (lane >> 2) + 8 * hr] = x;
    }
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float x = csum[n][e];
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        x += __shfl_xor_sync(0xffffffffu, x, 8);
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        if (lane < 4) sm.part[4 + (warp & 3)][c0 + 8 * n + 2 * lane + e] = -x;
      }
  }
  cp_async_wait<1>();  // H0, dE
  __syncthreads();
  // ---- 64 x 128 products: rows [r0, +16), columns [d0, +32)
  const int d0 = 32 * (warp >> 2);
  float acc[4][4], acc2[4][4];
  auto zero = [&](float (&x)[4][4]) {
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[n][e] = 0.f;
  };
  // acc += A (rows r0, K = 128 over `ld`-strided a) * Bt^T, Bt stored [n][k] (the H0^T / dH1^T forms)
  auto mm_abt = [&](float (&x)[4][4], uint32_t sa, uint32_t sbt) {
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(a, frag_a(sa, kS128, r0, 16 * kk, lane));
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t b[4];
        ldsm_x4(b, frag_bt(sbt, kS128, d0 + 16 * np, 16 * kk, lane));
        mma_bf16(x[2 * np], a, b[0], b[1]);
        mma_bf16(x[2 * np + 1], a, b[2], b[3]);
      }
    }
  };
  // acc += A (rows r0, K = 128) * B, B stored [k][n] (128 rows)
  auto mm_ab = [&](float (&x)[4][4], uint32_t sa, uint32_t sb) {
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(a, frag_a(sa, kS128, r0, 16 * kk, lane));
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t b[4];
        ldsm_x4_t(b, frag_b(sb, kS128, 16 * kk, d0 + 16 * np, lane));
        mma_bf16(x[2 * np], a, b[0], b[1]);
        mma_bf16(x[2 * np + 1], a, b[2], b[3]);
      }
    }
  };
  // dq = scale e^gamma dO H0^T + DG K
  zero(acc);
  zero(acc2);
  mm_abt(acc, sdO, sH0);
#pragma unroll
  for (int kk = 0; kk < kC / 16; ++kk) {
    uint32_t a[4];
    ldsm_x4(a, frag_a(sDG, kS64, r0, 16 * kk, lane));
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t b[4];
      ldsm_x4_t(b, frag_b(sK, kS128, 16 * kk, d0 + 16 * np, lane));
      mma_bf16(acc2[2 * np], a, b[0], b[1]);
      mma_bf16(acc2[2 * np + 1], a, b[2], b[3]);
    }
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = r0 + (lane >> 2) + 8 * hr;
    if (i < len) {
      const float m = p.scale * __expf(sm.gam[i]);
      __nv_bfloat16* row = p.dq + ((size_t)(t0 + i) * p.nh + h) * kD + d0;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int j = 8 * n + 2 * (lane & 3);
        *reinterpret_cast<uint32_t*>(row + j) =
            pack2(m * acc[n][2 * hr] + acc2[n][2 * hr], m * acc[n][2 * hr + 1] + acc2[n][2 * hr + 1]);
      }
    }
  }
  // dW = -dE H0^T
  zero(acc);
  mm_abt(acc, sdE, sH0);
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = r0 + (lane >> 2) + 8 * hr;
    if (i < len) {
      __nv_bfloat16* row = p.dW + ((size_t)(t0 + i) * p.nh + h) * kD + d0;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int j = 8 * n + 2 * (lane & 3);
        *reinterpret_cast<uint32_t*>(row + j) = pack2(-acc[n][2 * hr], -acc[n][2 * hr + 1]);
      }
    }
  }
  // dKa = w E dH1^T + DG^T Q
  cp_async_wait<0>();  // dH1
  __syncthreads();
  zero(acc);
  zero(acc2);
  mm_abt(acc, sE, sdH1);
#pragma unroll
  for (int kk = 0; kk < kC / 16; ++kk) {
    uint32_t a[4];
    ldsm_x4_t(a, frag_bt(sDG, kS64, 16 * kk, r0, lane));  // DG^T: DG stored [i][j]
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t b[4];
      ldsm_x4_t(b, frag_b(sQ, kS128, 16 * kk, d0 + 16 * np, lane));
      mma_bf16(acc2[2 * np], a, b[0], b[1]);
      mma_bf16(acc2[2 * np + 1], a, b[2], b[3]);
    }
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = r0 + (lane >> 2) + 8 * hr;
    if (i < len) {
      const float w = __expf(g_last - sm.gam[i]);
      float* row = p.dKa + ((size_t)(t0 + i) * p.nh + h) * kD + d0;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int j = 8 * n + 2 * (lane & 3);
        *reinterpret_cast<float2*>(row + j) =
            make_float2(w * acc[n][2 * hr] + acc2[n][2 * hr], w * acc[n][2 * hr + 1] + acc2[n][2 * hr + 1]);
      }
    }
  }
  // dgam: scale e^gamma_i <dO_i, (Q H0)_i> and the w_i <(K dH1)_i, E_i> terms
  zero(acc);
  zero(acc2);
  mm_ab(acc, sQ, sH0);
  mm_ab(acc2, sK, sdH1);
  {
    float rq[2] = {0.f, 0.f}, rk[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = r0 + (lane >> 2) + 8 * hr;
        const int j = d0 + 8 * n + 2 * (lane & 3);
        const float2 dd = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.dO[i * kS128 + j]));
        const float2 ee = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.E[i * kS128 + j]));
        rq[hr] += acc[n][2 * hr] * dd.x + acc[n][2 * hr + 1] * dd.y;
        rk[hr] += acc2[n][2 * hr] * ee.x + acc2[n][2 * hr + 1] * ee.y;
      }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = r0 + (lane >> 2) + 8 * hr;
      const float q_ = quad_sum(rq[hr]), k_ = quad_sum(rk[hr]);
      if ((lane & 3) == 0 && i < len) {
        const float w = __expf(g_last - sm.gam[i]);
        sm.part[8 + (warp >> 2)][i] = p.scale * __expf(sm.gam[i]) * q_ - w * k_;
        sm.lw[warp >> 2][i] = w * k_;
      }
    }
    // e^gamma_last <dH1, H0>: this thread's share of the 128 x 128 products
    float t = 0.f;
    for (int e = tid; e < kD * kD / 2; e += nt) {
      const int rr = e >> 6, cc = (e & 63) * 2;
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.H0[rr * kS128 + cc]));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.dH1[rr * kS128 + cc]));
      t += a.x * b.x + a.y * b.y;
    }
    float x = t;
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) sm.tw[warp] = x;
  }
  __syncthreads();
  if (warp == 0) {
    // the gamma_last terms: lane l adds rows l and l + 32 of the four slots
    // and warp l's <dH1, H0> share, then a fixed butterfly over the lanes
    float last = 0.f, t = lane < kLocalThreads / 32 ? sm.tw[lane] : 0.f;
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) last += sm.lw[sl][lane] + sm.lw[sl][lane + 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      last += __shfl_xor_sync(0xffffffffu, last, o);
      t += __shfl_xor_sync(0xffffffffu, t, o);
    }
    if (lane == 0) sm.last = last + __expf(g_last) * t;
  }
  if (tid < kC) {
    float d = 0.f;
    for (int sl = 0; sl < 12; ++sl) d += sm.part[sl][tid];
    sm.dgs[tid] = d;
  }
  __syncthreads();
  if (tid < len) p.dgam[(size_t)h * p.total + t0 + tid] = sm.dgs[tid] + (tid == len - 1 ? sm.last : 0.f);
}

// ============================================================== Kimi Delta backward: local, with the states
// Per (chunk, head), with B = e^gamma per channel, QB = Q o B, KC = K o e^(gamma_last - gamma):
//     dQB = scale dO H0^T       ->  dQa = dQB o B,            dgam += dQB o QB
//     dW  = -dE H0^T
//     dKC = E dH1^T             ->  dKa = dKC o e^(gamma_last - gamma),  dgam -= dKC o KC,
//                                   dgam_last += sum_i dKC_i o KC_i
//     dgam_last += e^gamma_last o rowsum(dH1 o H0)
//     N   = lower(scale dO E^T) (the gradient of the masked q.k block, to the workspace)
struct KdaLocalHSmem {
  __nv_bfloat16 dO[kC * kS128];
  __nv_bfloat16 dE[kC * kS128];
  __nv_bfloat16 E[kC * kS128];
  __nv_bfloat16 QB[kC * kS128];
  __nv_bfloat16 KC[kC * kS128];
  __nv_bfloat16 H0[kD * kS128];
  __nv_bfloat16 dH1[kD * kS128];
  float G[kC * kG];  // gamma per channel
  float last[kD];    // the gamma_last terms per channel
  float lc[4][kD];   // their column partials from the four row groups, added in a fixed order
  float tot[4 * kD];               // scratch of the channel running sums
};
static_assert(sizeof(KdaLocalHSmem) <= 227 * 1024, "fits one SM");

__global__ void __launch_bounds__(kLocalThreads) kda_bwd_local_h_kernel(GdnParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  KdaLocalHSmem& sm = *reinterpret_cast<KdaLocalHSmem*>(smem_raw);
  constexpr int nt = kLocalThreads;
  grid_dependency_wait();
  const int c = blockIdx.x, h = blockIdx.y;
  const int n_chunks = __ldcg(p.hdr);
  const int4 ch = p.chunks[c];
  if (c >= n_chunks) return;
  const int len = chunk_len(ch, p.total);
  if (len <= 0) return;  // only with a boundary list that breaks its rules
  const int t0 = ch.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sdO = smem_u32(sm.dO), sdE = smem_u32(sm.dE), sE = smem_u32(sm.E), sH0 = smem_u32(sm.H0),
                 sdH1 = smem_u32(sm.dH1);
  // Three copy groups, waited for in the order the products need them:
  // dO, E and the gates (gamma, N); H0, dE, QB (dQB, dW); dH1, KC (dKC).
  load_rows128(sdO, p.dO, t0, len, h, p.nh, tid, nt);
  load_rows128(sE, p.E, t0, len, h, p.nh, tid, nt);
  for (int e = tid; e < kC * 32; e += nt) {
    const int r = e >> 5, cc = (e & 31) * 4;
    const bool ok = r < len;
    cp_async16(smem_u32(&sm.G[r * kG + cc]), p.g + ((size_t)(t0 + (ok ? r : 0)) * p.nh + h) * kD + cc, ok);
  }
  cp_async_commit();
  const __nv_bfloat16* h0 = p.H0 + ((size_t)c * p.nh + h) * (kD * kD);
  const __nv_bfloat16* d1 = p.dH1 + ((size_t)c * p.nh + h) * (kD * kD);
  for (int e = tid; e < kD * 16; e += nt) {
    const int r = e >> 4, cc = (e & 15) * 8;
    cp_async16(sH0 + 2u * (uint32_t)(r * kS128 + cc), h0 + r * kD + cc, true);
  }
  load_rows128(sdE, p.dE, t0, len, h, p.nh, tid, nt);
  load_rows128(smem_u32(sm.QB), p.QB, t0, len, h, p.nh, tid, nt);
  cp_async_commit();
  for (int e = tid; e < kD * 16; e += nt) {
    const int r = e >> 4, cc = (e & 15) * 8;
    cp_async16(sdH1 + 2u * (uint32_t)(r * kS128 + cc), d1 + r * kD + cc, true);
  }
  load_rows128(smem_u32(sm.KC), p.KC, t0, len, h, p.nh, tid, nt);
  cp_async_commit();
  cp_async_wait<2>();
  __syncthreads();
  chan_running_sum(sm.G, sm.tot, tid);  // gamma per channel
  const int r0 = 16 * (warp & 3);
  // ---- N = lower(scale dO E^T): rows [r0, +16) x columns [c0, +16)
  {
    const int c0 = 16 * (warp >> 2);
    float s1[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) s1[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t a[4], b[4];
      ldsm_x4(a, frag_a(sdO, kS128, r0, 16 * kk, lane));
      ldsm_x4(b, frag_bt(sE, kS128, c0, 16 * kk, lane));
      mma_bf16(s1[0], a, b[0], b[1]);
      mma_bf16(s1[1], a, b[2], b[3]);
    }
    float* nw = p.Nw + ((size_t)c * p.nh + h) * (kC * kC);
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = r0 + (lane >> 2) + 8 * hr;
        const int j = c0 + 8 * n + 2 * (lane & 3);
        *reinterpret_cast<float2*>(nw + i * kC + j) =
            make_float2(j <= i ? p.scale * s1[n][2 * hr] : 0.f, j + 1 <= i ? p.scale * s1[n][2 * hr + 1] : 0.f);
      }
  }
  cp_async_wait<1>();  // H0, dE, QB
  __syncthreads();
  // ---- 64 x 128 products: rows [r0, +16), columns [d0, +32)
  const int d0 = 32 * (warp >> 2);
  float acc[4][4], dg[2][4][2];
  auto zero = [&](float (&x)[4][4]) {
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[n][e] = 0.f;
  };
  // acc += A (rows r0, K = 128) * Bt^T, Bt stored [n][k] (the H0^T / dH1^T forms)
  auto mm_abt = [&](float (&x)[4][4], uint32_t sa, uint32_t sbt) {
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(a, frag_a(sa, kS128, r0, 16 * kk, lane));
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t b[4];
        ldsm_x4(b, frag_bt(sbt, kS128, d0 + 16 * np, 16 * kk, lane));
        mma_bf16(x[2 * np], a, b[0], b[1]);
        mma_bf16(x[2 * np + 1], a, b[2], b[3]);
      }
    }
  };
  // dQB = scale dO H0^T
  zero(acc);
  mm_abt(acc, sdO, sH0);
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = r0 + (lane >> 2) + 8 * hr;
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const int j = d0 + 8 * n + 2 * (lane & 3);
      const float a0 = p.scale * acc[n][2 * hr], a1 = p.scale * acc[n][2 * hr + 1];
      const float2 qb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.QB[i * kS128 + j]));
      dg[hr][n][0] = a0 * qb.x;
      dg[hr][n][1] = a1 * qb.y;
      if (i < len)
        *reinterpret_cast<float2*>(p.dQa + ((size_t)(t0 + i) * p.nh + h) * kD + j) =
            make_float2(a0 * __expf(sm.G[i * kG + j]), a1 * __expf(sm.G[i * kG + j + 1]));
    }
  }
  // dW = -dE H0^T
  zero(acc);
  mm_abt(acc, sdE, sH0);
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = r0 + (lane >> 2) + 8 * hr;
    if (i < len) {
      __nv_bfloat16* row = p.dW + ((size_t)(t0 + i) * p.nh + h) * kD + d0;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int j = 8 * n + 2 * (lane & 3);
        *reinterpret_cast<uint32_t*>(row + j) = pack2(-acc[n][2 * hr], -acc[n][2 * hr + 1]);
      }
    }
  }
  cp_async_wait<0>();  // dH1, KC
  __syncthreads();
  if (tid < kD) {  // e^gamma_last rowsum(dH1 o H0) of the channel (row tid of H)
    float d = 0.f;
    for (int v = 0; v < kD; v += 2) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.H0[tid * kS128 + v]));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.dH1[tid * kS128 + v]));
      d += a.x * b.x + a.y * b.y;
    }
    sm.last[tid] = d * __expf(sm.G[(len - 1) * kG + tid]);  // this thread adds the rest later
  }
  // dKC = E dH1^T
  zero(acc);
  mm_abt(acc, sE, sdH1);
  float colp[4][2];  // this thread's part of sum_i dKC_i o KC_i, per column
#pragma unroll
  for (int n = 0; n < 4; ++n) colp[n][0] = colp[n][1] = 0.f;
  const float* glast = &sm.G[(len - 1) * kG];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = r0 + (lane >> 2) + 8 * hr;
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const int j = d0 + 8 * n + 2 * (lane & 3);
      const float a0 = acc[n][2 * hr], a1 = acc[n][2 * hr + 1];
      const float2 kc = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.KC[i * kS128 + j]));
      dg[hr][n][0] -= a0 * kc.x;
      dg[hr][n][1] -= a1 * kc.y;
      if (i < len) {
        colp[n][0] += a0 * kc.x;
        colp[n][1] += a1 * kc.y;
        *reinterpret_cast<float2*>(p.dKa + ((size_t)(t0 + i) * p.nh + h) * kD + j) =
            make_float2(a0 * __expf(glast[j] - sm.G[i * kG + j]), a1 * __expf(glast[j + 1] - sm.G[i * kG + j + 1]));
      }
    }
  }
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float x = colp[n][e];
      x += __shfl_xor_sync(0xffffffffu, x, 4);
      x += __shfl_xor_sync(0xffffffffu, x, 8);
      x += __shfl_xor_sync(0xffffffffu, x, 16);
      if (lane < 4) sm.lc[warp & 3][d0 + 8 * n + 2 * lane + e] = x;
    }
  __syncthreads();
  if (tid < kD) sm.last[tid] += ((sm.lc[0][tid] + sm.lc[1][tid]) + sm.lc[2][tid]) + sm.lc[3][tid];
  __syncthreads();
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = r0 + (lane >> 2) + 8 * hr;
    if (i < len) {
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int j = d0 + 8 * n + 2 * (lane & 3);
        float x0 = dg[hr][n][0], x1 = dg[hr][n][1];
        if (i == len - 1) {
          x0 += sm.last[j];
          x1 += sm.last[j + 1];
        }
        *reinterpret_cast<float2*>(p.dgam + ((size_t)(t0 + i) * p.nh + h) * kD + j) = make_float2(x0, x1);
      }
    }
  }
}

// Xb = X in bf16 and XT = X transposed (fp32, row stride kS4), by the 512
// threads of a local CTA.  A warp takes an 8 x 4 block per round (row = lane
// % 8, column = lane / 8): its reads of X fall in 32 different banks, and
// its writes of XT at most two to a bank.
__device__ __forceinline__ void wy_copy_x(const float* X, __nv_bfloat16* Xb, float* XT, int tid) {
#pragma unroll 4
  for (int e = tid; e < kC * kC; e += kLocalThreads) {
    const int blk = e >> 5, l = e & 31;
    const int i = 8 * (blk >> 4) + (l & 7), j = 4 * (blk & 15) + (l >> 3);
    const float x = X[i * kS4 + j];
    Xb[i * kS64 + j] = __float2bfloat16_rn(x);
    XT[j * kS4 + i] = x;
  }
}

// dA = strictly-lower(-X^T dX X^T) for the unit lower-triangular X of a
// chunk, in fp32, by the 16 warps of a local CTA:
//     Y = dX X^T  (into Y),   dA = -X^T Y  (into dA, zero on and above the diagonal).
// dXT = dX transposed and XT = X transposed, [m][i] with row stride kS4; X
// [m][i], Y [m][j] with kS4; dA with kSF.  Warp w owns four columns j0 .. j0
// + 3 and lane l the rows 2l, 2l + 1.  X[j][m] = 0 for m > j, so Y's sums
// stop at m = j0 + 3; X[m][i] = 0 for m < i and only i > j is kept, so dA's
// sums start at m = j0 + 1.  The terms left out multiply exact zeros, so the
// sums are the full ones, term for term in the same order.  The column
// blocks are dealt so that the four warps of each scheduler have equal loop
// lengths.
__device__ __forceinline__ void wy_grad_a(const float* dXT, const float* XT, const float* X, float* Y, float* dA,
                                          int warp, int lane) {
  const int k = warp >> 2, sch = warp & 3;
  const int cb = k == 0 ? sch : (k == 1 ? 7 - sch : (k == 2 ? 8 + sch : 15 - sch));
  const int j0 = 4 * cb, i0 = 2 * lane;
  float y[2][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) y[a][b] = 0.f;
#pragma unroll 4
  for (int m = 0; m < j0 + 4; ++m) {
    const float2 xa = *reinterpret_cast<const float2*>(&dXT[m * kS4 + i0]);  // dX[i0 + a][m]
    const float4 xb = *reinterpret_cast<const float4*>(&XT[m * kS4 + j0]);   // X[j0 + b][m], one broadcast
    const float av[2] = {xa.x, xa.y}, bv[4] = {xb.x, xb.y, xb.z, xb.w};
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) y[a][b] = fmaf(av[a], bv[b], y[a][b]);
  }
#pragma unroll
  for (int a = 0; a < 2; ++a)
    *reinterpret_cast<float4*>(&Y[(i0 + a) * kS4 + j0]) = make_float4(y[a][0], y[a][1], y[a][2], y[a][3]);
  __syncthreads();
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) y[a][b] = 0.f;
#pragma unroll 4
  for (int m = j0 + 1; m < kC; ++m) {
    const float2 xa = *reinterpret_cast<const float2*>(&X[m * kS4 + i0]);  // X[m][i0 + a]
    const float4 xb = *reinterpret_cast<const float4*>(&Y[m * kS4 + j0]);  // Y[m][j0 + b], one broadcast
    const float av[2] = {xa.x, xa.y}, bv[4] = {xb.x, xb.y, xb.z, xb.w};
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) y[a][b] = fmaf(av[a], bv[b], y[a][b]);
  }
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) dA[(i0 + a) * kSF + j0 + b] = j0 + b < i0 + a ? -y[a][b] : 0.f;
}

// ============================================================== backward: local, the WY factors
// Per (chunk, head), from K, V, dE, dW (A and X = (I + A)^-1 recomputed):
//     dX  = (dE V^T) diag(beta) + (dW K^T) diag(beta e^gamma)
//     dA  = strictly-lower(-X^T dX X^T),  M = diag(beta) (dA o Gamma)
//     dVb = X^T dE,  dKb = X^T dW
//     dv  = diag(beta) dVb
//     dk  = dKa + diag(beta e^gamma) dKb + M K + M^T K
//     dbeta_i = sum_j dA_ij Gamma_ij <k_i, k_j> + <dVb_i, v_i> + e^gamma_i <dKb_i, k_i>
//     dgam_i += rowsum_i - colsum_i of M o (K K^T) + beta_i e^gamma_i <dKb_i, k_i>
//     dg  = reverse running sum of dgam over the chunk
struct LocalWySmem {
  __nv_bfloat16 K[kC * kS128];
  __nv_bfloat16 V[kC * kS128];
  __nv_bfloat16 dE[kC * kS128];
  __nv_bfloat16 dW[kC * kS128];
  float A[kC * kSF];    // A, then dA, then dA o Gamma o KK
  float KK[kC * kSF];   // K K^T, then M o KK
  float X[kC * kS4];    // (I + A)^-1
  float XT[kC * kS4];   // its transpose
  float dXT[kC * kS4];  // dX, transposed
  float Y[kC * kS4];    // dX X^T
  alignas(16) float R[3 * 256];
  __nv_bfloat16 Xb[kC * kS64];
  __nv_bfloat16 M[kC * kS64];
  float gam[kC];
  float bet[kC];
  float dgs[kC];
  float dbs[kC];
  float pb[4][kC];  // row partials of dbeta and dgam from the four column groups, added in a fixed order
  float pg[4][kC];
};
static_assert(sizeof(LocalWySmem) <= 227 * 1024, "fits one SM");

__global__ void __launch_bounds__(kLocalThreads) gdn_bwd_local_wy_kernel(GdnParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  LocalWySmem& sm = *reinterpret_cast<LocalWySmem*>(smem_raw);
  constexpr int nt = kLocalThreads;
  grid_dependency_wait();
  const int c = blockIdx.x, h = blockIdx.y;
  // (both loads in flight at once: the table entry is in bounds for every
  // c < max_chunks, and ignored past the number of chunks)
  const int n_chunks = __ldcg(p.hdr);
  const int4 ch = p.chunks[c];
  if (c >= n_chunks) return;
  const int len = chunk_len(ch, p.total);
  if (len <= 0) return;  // only with a boundary list that breaks its rules
  const int t0 = ch.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sK = smem_u32(sm.K), sV = smem_u32(sm.V), sdE = smem_u32(sm.dE), sdW = smem_u32(sm.dW),
                 sXb = smem_u32(sm.Xb), sM = smem_u32(sm.M);
  load_rows128(sK, p.k, t0, len, h, p.nh, tid, nt);
  load_rows128(sV, p.v, t0, len, h, p.nh, tid, nt);
  load_rows128(sdE, p.dE, t0, len, h, p.nh, tid, nt);
  load_rows128(sdW, p.dW, t0, len, h, p.nh, tid, nt);
  cp_async_commit();
  if (tid < kC) {
    const bool ok = tid < len;
    sm.gam[tid] = ok ? p.gam[(size_t)h * p.total + t0 + tid] : 0.f;
    sm.bet[tid] = ok ? p.beta[(size_t)(t0 + tid) * p.nh + h] : 0.f;
    sm.dgs[tid] = ok ? p.dgam[(size_t)h * p.total + t0 + tid] : 0.f;
    sm.dbs[tid] = 0.f;
  }
  cp_async_wait<0>();
  __syncthreads();
  const int r0 = 16 * (warp & 3);
  // ---- K K^T (rows [r0, +16), columns [c0, +32)): A and KK
  {
    const int c0 = 16 * (warp >> 2);
    float s[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(a, frag_a(sK, kS128, r0, 16 * kk, lane));
#pragma unroll
      for (int np = 0; np < 1; ++np) {
        uint32_t b[4];
        ldsm_x4(b, frag_bt(sK, kS128, c0 + 16 * np, 16 * kk, lane));
        mma_bf16(s[2 * np], a, b[0], b[1]);
        mma_bf16(s[2 * np + 1], a, b[2], b[3]);
      }
    }
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = r0 + (lane >> 2) + 8 * hr;
          const int j = c0 + 8 * n + 2 * (lane & 3) + e;
          const float kk_ = s[n][2 * hr + e];
          sm.KK[i * kSF + j] = kk_;
          sm.A[i * kSF + j] = j < i ? sm.bet[i] * __expf(sm.gam[i] - sm.gam[j]) * kk_ : 0.f;
        }
  }
  __syncthreads();
  wy_inverse<kS4, kLocalThreads>(sm.A, sm.X, sm.R, tid);
  // ---- Xb = bf16 X, XT; dX = (dE V^T) diag(beta) + (dW K^T) diag(beta e^gamma)
  wy_copy_x(sm.X, sm.Xb, sm.XT, tid);
  {
    const int c0 = 16 * (warp >> 2);
    float pv[2][4], pk[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) pv[n][e] = pk[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t ae[4], aw[4];
      ldsm_x4(ae, frag_a(sdE, kS128, r0, 16 * kk, lane));
      ldsm_x4(aw, frag_a(sdW, kS128, r0, 16 * kk, lane));
#pragma unroll
      for (int np = 0; np < 1; ++np) {
        uint32_t bv[4], bk[4];
        ldsm_x4(bv, frag_bt(sV, kS128, c0 + 16 * np, 16 * kk, lane));
        ldsm_x4(bk, frag_bt(sK, kS128, c0 + 16 * np, 16 * kk, lane));
        mma_bf16(pv[2 * np], ae, bv[0], bv[1]);
        mma_bf16(pv[2 * np + 1], ae, bv[2], bv[3]);
        mma_bf16(pk[2 * np], aw, bk[0], bk[1]);
        mma_bf16(pk[2 * np + 1], aw, bk[2], bk[3]);
      }
    }
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = r0 + (lane >> 2) + 8 * hr;
          const int j = c0 + 8 * n + 2 * (lane & 3) + e;
          const float bj = sm.bet[j];
          sm.dXT[j * kS4 + i] = pv[n][2 * hr + e] * bj + pk[n][2 * hr + e] * bj * __expf(sm.gam[j]);
        }
  }
  __syncthreads();
  // ---- Y = dX X^T, then dA = -X^T Y, strictly lower (fp32)
  wy_grad_a(sm.dXT, sm.XT, sm.X, sm.Y, sm.A, warp, lane);
  __syncthreads();
  // ---- M = diag(beta) (dA o Gamma) (bf16); in place, A becomes dA o Gamma o KK
  // (its row sums go to dbeta) and KK becomes M o KK (row minus column sums
  // to dgam)
  for (int e = tid; e < kC * kC / 2; e += nt) {
    const int i = e >> 5, j = (e & 31) * 2;
    const float g0 = j < i ? __expf(sm.gam[i] - sm.gam[j]) : 0.f;
    const float g1 = j + 1 < i ? __expf(sm.gam[i] - sm.gam[j + 1]) : 0.f;
    const float a0 = sm.A[i * kSF + j] * g0, a1 = sm.A[i * kSF + j + 1] * g1;
    const float k0 = sm.KK[i * kSF + j], k1 = sm.KK[i * kSF + j + 1];
    const float m0 = sm.bet[i] * a0, m1 = sm.bet[i] * a1;
    *reinterpret_cast<uint32_t*>(&sm.M[i * kS64 + j]) = pack2(m0, m1);
    sm.A[i * kSF + j] = a0 * k0;
    sm.A[i * kSF + j + 1] = a1 * k1;
    sm.KK[i * kSF + j] = m0 * k0;
    sm.KK[i * kSF + j + 1] = m1 * k1;
  }
  __syncthreads();
  if (tid < kC) {
    float rb = 0.f, rg = 0.f;
    for (int j = 0; j < kC; ++j) {
      rb += sm.A[tid * kSF + j];
      rg += sm.KK[tid * kSF + j];
    }
    sm.dbs[tid] += rb;
    sm.dgs[tid] += rg;
  }
  __syncthreads();
  if (tid < kC) {
    float cg = 0.f;
    for (int i = 0; i < kC; ++i) cg += sm.KK[i * kSF + tid];
    sm.dgs[tid] -= cg;
  }
  __syncthreads();
  // ---- 64 x 128 products, rows [r0, +16) x columns [d0, +32)
  const int d0 = 32 * (warp >> 2);
  // this thread's part of dKa, loaded now for the dk store at the end.  A
  // row past the chunk reads row 0 instead (never used): no select on the
  // loaded value, so the warp does not wait for it here.
  float2 dka[2][4];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = r0 + (lane >> 2) + 8 * hr;
    const size_t off = ((size_t)(t0 + (i < len ? i : 0)) * p.nh + h) * kD + d0;
#pragma unroll
    for (int n = 0; n < 4; ++n)
      dka[hr][n] = *reinterpret_cast<const float2*>(p.dKa + off + 8 * n + 2 * (lane & 3));
  }
  float cv[4][4], ck[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) cv[n][e] = ck[n][e] = 0.f;
  // dVb = X^T dE, dKb = X^T dW
#pragma unroll
  for (int kk = 0; kk < kC / 16; ++kk) {
    uint32_t a[4];
    ldsm_x4_t(a, frag_bt(sXb, kS64, 16 * kk, r0, lane));  // X^T: X stored [i][j]
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t be[4], bw[4];
      ldsm_x4_t(be, frag_b(sdE, kS128, 16 * kk, d0 + 16 * np, lane));
      ldsm_x4_t(bw, frag_b(sdW, kS128, 16 * kk, d0 + 16 * np, lane));
      mma_bf16(cv[2 * np], a, be[0], be[1]);
      mma_bf16(cv[2 * np + 1], a, be[2], be[3]);
      mma_bf16(ck[2 * np], a, bw[0], bw[1]);
      mma_bf16(ck[2 * np + 1], a, bw[2], bw[3]);
    }
  }
  // dv, and the <dVb, v>, <dKb, k> row sums; dk starts as diag(beta e^gamma) dKb
  {
    float rv[2] = {0.f, 0.f}, rk[2] = {0.f, 0.f};
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = r0 + (lane >> 2) + 8 * hr;
      const float bi = sm.bet[i], be = bi * __expf(sm.gam[i]);
      __nv_bfloat16* row = p.dv + ((size_t)(t0 + i) * p.nh + h) * kD + d0;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int j = 8 * n + 2 * (lane & 3);
        const float2 vv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.V[i * kS128 + d0 + j]));
        const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.K[i * kS128 + d0 + j]));
        rv[hr] += cv[n][2 * hr] * vv.x + cv[n][2 * hr + 1] * vv.y;
        rk[hr] += ck[n][2 * hr] * kv.x + ck[n][2 * hr + 1] * kv.y;
        if (i < len) *reinterpret_cast<uint32_t*>(row + j) = pack2(bi * cv[n][2 * hr], bi * cv[n][2 * hr + 1]);
        ck[n][2 * hr] *= be;
        ck[n][2 * hr + 1] *= be;
      }
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = r0 + (lane >> 2) + 8 * hr;
      const float v_ = quad_sum(rv[hr]), k_ = quad_sum(rk[hr]);
      if ((lane & 3) == 0) {
        const float eg = __expf(sm.gam[i]);
        sm.pb[warp >> 2][i] = v_ + eg * k_;
        sm.pg[warp >> 2][i] = sm.bet[i] * eg * k_;
      }
    }
  }
  // dk += M K + M^T K (+ dKa)
#pragma unroll
  for (int kk = 0; kk < kC / 16; ++kk) {
    uint32_t am[4], at[4];
    ldsm_x4(am, frag_a(sM, kS64, r0, 16 * kk, lane));
    ldsm_x4_t(at, frag_bt(sM, kS64, 16 * kk, r0, lane));  // M^T
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t b[4];
      ldsm_x4_t(b, frag_b(sK, kS128, 16 * kk, d0 + 16 * np, lane));
      mma_bf16(ck[2 * np], am, b[0], b[1]);
      mma_bf16(ck[2 * np + 1], am, b[2], b[3]);
      mma_bf16(ck[2 * np], at, b[0], b[1]);
      mma_bf16(ck[2 * np + 1], at, b[2], b[3]);
    }
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = r0 + (lane >> 2) + 8 * hr;
    if (i < len) {
      const size_t off = ((size_t)(t0 + i) * p.nh + h) * kD + d0;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int j = 8 * n + 2 * (lane & 3);
        *reinterpret_cast<uint32_t*>(p.dk + off + j) =
            pack2(ck[n][2 * hr] + dka[hr][n].x, ck[n][2 * hr + 1] + dka[hr][n].y);
      }
    }
  }
  __syncthreads();
  if (tid < kC) {
    sm.dbs[tid] += ((sm.pb[0][tid] + sm.pb[1][tid]) + sm.pb[2][tid]) + sm.pb[3][tid];
    sm.dgs[tid] += ((sm.pg[0][tid] + sm.pg[1][tid]) + sm.pg[2][tid]) + sm.pg[3][tid];
  }
  __syncthreads();
  // dbeta, and dg = reverse running sum of dgam (one warp, two tokens per lane)
  if (tid < len) p.dbeta[(size_t)(t0 + tid) * p.nh + h] = sm.dbs[tid];
  if (warp == 0) {
    const int i0 = 62 - 2 * lane;  // lane 0 takes the last two tokens
    const float a1 = sm.dgs[i0 + 1], a0 = sm.dgs[i0];
    const float s2 = a0 + a1;
    float incl = s2;
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const float ex = incl - s2;  // sum over tokens after i0 + 1
    if (i0 + 1 < len) p.dg[(size_t)(t0 + i0 + 1) * p.nh + h] = ex + a1;
    if (i0 < len) p.dg[(size_t)(t0 + i0) * p.nh + h] = ex + a1 + a0;
  }
}
// ============================================================== Kimi Delta backward: local, the WY factors
// Per (chunk, head), from K, V, dE, dW and the recomputation's X and A (unscaled):
//     dX  = (dE V^T + dW KB^T) diag(beta),   KB = K o e^gamma
//     dA  = strictly-lower(-X^T dX X^T),      M = diag(beta) dA   (to the workspace)
//     dVb = X^T dE,  XdW = X^T dW
//     dv  = diag(beta) dVb                                          (final)
//     dbeta_i = sum_j dA_ij Araw_ij + <dVb_i, v_i> + <XdW_i, KB_i>  (final)
//     dKa += diag(beta) XdW o e^gamma,  dgam += diag(beta) XdW o KB
struct KdaLocalWySmem {
  __nv_bfloat16 KB[kC * kS128];  // K, then K o e^gamma
  __nv_bfloat16 V[kC * kS128];
  __nv_bfloat16 dE[kC * kS128];
  __nv_bfloat16 dW[kC * kS128];
  float G[kC * kG];
  float X[kC * kS4];
  float XT[kC * kS4];
  float dXT[kC * kS4];
  float Y[kC * kS4];
  float A[kC * kSF];    // dA
  float Ar[kC * kSF];   // the unscaled A
  __nv_bfloat16 Xb[kC * kS64];
  float bet[kC];
  float dbs[kC];
  float pb[4][kC];  // row partials of dbeta from the four column groups, added in a fixed order
  float tot[4 * kD];               // scratch of the channel running sums
};
static_assert(sizeof(KdaLocalWySmem) <= 227 * 1024, "fits one SM");

__global__ void __launch_bounds__(kLocalThreads) kda_bwd_local_wy_kernel(GdnParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  KdaLocalWySmem& sm = *reinterpret_cast<KdaLocalWySmem*>(smem_raw);
  constexpr int nt = kLocalThreads;
  grid_dependency_wait();
  const int c = blockIdx.x, h = blockIdx.y;
  const int n_chunks = __ldcg(p.hdr);
  const int4 ch = p.chunks[c];
  if (c >= n_chunks) return;
  const int len = chunk_len(ch, p.total);
  if (len <= 0) return;  // only with a boundary list that breaks its rules
  const int t0 = ch.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sKB = smem_u32(sm.KB), sV = smem_u32(sm.V), sdE = smem_u32(sm.dE), sdW = smem_u32(sm.dW),
                 sXb = smem_u32(sm.Xb);
  load_rows128(sKB, p.k, t0, len, h, p.nh, tid, nt);
  load_rows128(sV, p.v, t0, len, h, p.nh, tid, nt);
  load_rows128(sdE, p.dE, t0, len, h, p.nh, tid, nt);
  load_rows128(sdW, p.dW, t0, len, h, p.nh, tid, nt);
  for (int e = tid; e < kC * 32; e += nt) {
    const int r = e >> 5, cc = (e & 31) * 4;
    const bool ok = r < len;
    cp_async16(smem_u32(&sm.G[r * kG + cc]), p.g + ((size_t)(t0 + (ok ? r : 0)) * p.nh + h) * kD + cc, ok);
  }
  {
    const size_t base = ((size_t)c * p.nh + h) * (kC * kC);
    for (int e = tid; e < kC * 16; e += nt) {  // X and the unscaled A, 16 pieces of 4 floats per row
      const int r = e >> 4, cc = (e & 15) * 4;
      cp_async16(smem_u32(&sm.X[r * kS4 + cc]), p.Xw + base + r * kC + cc, true);
    }
  }
  cp_async_commit();
  if (tid < kC) {
    sm.bet[tid] = tid < len ? p.beta[(size_t)(t0 + tid) * p.nh + h] : 0.f;
    sm.dbs[tid] = 0.f;
  }
  {
    const float* ar = p.Araw + ((size_t)c * p.nh + h) * (kC * kC);
    static_assert(kC * kC % nt == 0, "whole rounds");
    float v[kC * kC / nt];  // all loads in flight before the first store
#pragma unroll
    for (int k = 0; k < kC * kC / nt; ++k) v[k] = ar[tid + k * nt];
#pragma unroll
    for (int k = 0; k < kC * kC / nt; ++k) {
      const int e = tid + k * nt;
      sm.Ar[(e >> 6) * kSF + (e & 63)] = v[k];
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  chan_running_sum(sm.G, sm.tot, tid);  // gamma per channel
  // KB = K o e^gamma in place; Xb, XT
  for (int e = tid; e < kC * kD / 2; e += nt) {
    const int i = e >> 6, cc = (e & 63) * 2;
    const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.KB[i * kS128 + cc]));
    *reinterpret_cast<uint32_t*>(&sm.KB[i * kS128 + cc]) =
        pack2(kv.x * __expf(sm.G[i * kG + cc]), kv.y * __expf(sm.G[i * kG + cc + 1]));
  }
  wy_copy_x(sm.X, sm.Xb, sm.XT, tid);
  __syncthreads();
  const int r0 = 16 * (warp & 3);
  // ---- dX = (dE V^T + dW KB^T) diag(beta): rows [r0, +16) x columns [c0, +16), stored transposed
  {
    const int c0 = 16 * (warp >> 2);
    float pv[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) pv[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t ae[4], aw[4], bv[4], bk[4];
      ldsm_x4(ae, frag_a(sdE, kS128, r0, 16 * kk, lane));
      ldsm_x4(aw, frag_a(sdW, kS128, r0, 16 * kk, lane));
      ldsm_x4(bv, frag_bt(sV, kS128, c0, 16 * kk, lane));
      ldsm_x4(bk, frag_bt(sKB, kS128, c0, 16 * kk, lane));
      mma_bf16(pv[0], ae, bv[0], bv[1]);
      mma_bf16(pv[1], ae, bv[2], bv[3]);
      mma_bf16(pv[0], aw, bk[0], bk[1]);
      mma_bf16(pv[1], aw, bk[2], bk[3]);
    }
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = r0 + (lane >> 2) + 8 * hr;
          const int j = c0 + 8 * n + 2 * (lane & 3) + e;
          sm.dXT[j * kS4 + i] = pv[n][2 * hr + e] * sm.bet[j];
        }
  }
  __syncthreads();
  // ---- Y = dX X^T, then dA = -X^T Y, strictly lower (fp32)
  wy_grad_a(sm.dXT, sm.XT, sm.X, sm.Y, sm.A, warp, lane);
  __syncthreads();
  // ---- M = diag(beta) dA to the workspace; sum_j dA_ij Araw_ij into dbeta
  {
    float* mw = p.Mw + ((size_t)c * p.nh + h) * (kC * kC);
    for (int e = tid; e < kC * kC; e += nt) {
      const int i = e >> 6, j = e & 63;
      mw[e] = sm.bet[i] * sm.A[i * kSF + j];
    }
    if (tid < kC) {
      float rb = 0.f;
      for (int j = 0; j < kC; ++j) rb += sm.A[tid * kSF + j] * sm.Ar[tid * kSF + j];
      sm.dbs[tid] += rb;
    }
  }
  __syncthreads();  // dbs gets atomic adds below
  // ---- dVb = X^T dE, XdW = X^T dW: rows [r0, +16) x columns [d0, +32)
  const int d0 = 32 * (warp >> 2);
  // this thread's dKa and dgam elements, read now so that the reads overlap
  // the products (the epilogue updates them in place)
  float2 kav[2][4], gav[2][4];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    // (a row past the chunk reads row 0 instead, never used: no select on the
    // loaded values, so the warp does not wait for them here)
    const int i = r0 + (lane >> 2) + 8 * hr;
    const size_t off = ((size_t)(t0 + (i < len ? i : 0)) * p.nh + h) * kD + d0;
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const int j = 8 * n + 2 * (lane & 3);
      kav[hr][n] = *reinterpret_cast<const float2*>(p.dKa + off + j);
      gav[hr][n] = *reinterpret_cast<const float2*>(p.dgam + off + j);
    }
  }
  float cv[4][4], ck[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) cv[n][e] = ck[n][e] = 0.f;
#pragma unroll
  for (int kk = 0; kk < kC / 16; ++kk) {
    uint32_t a[4];
    ldsm_x4_t(a, frag_bt(sXb, kS64, 16 * kk, r0, lane));  // X^T: X stored [i][j]
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t be[4], bw[4];
      ldsm_x4_t(be, frag_b(sdE, kS128, 16 * kk, d0 + 16 * np, lane));
      ldsm_x4_t(bw, frag_b(sdW, kS128, 16 * kk, d0 + 16 * np, lane));
      mma_bf16(cv[2 * np], a, be[0], be[1]);
      mma_bf16(cv[2 * np + 1], a, be[2], be[3]);
      mma_bf16(ck[2 * np], a, bw[0], bw[1]);
      mma_bf16(ck[2 * np + 1], a, bw[2], bw[3]);
    }
  }
  {
    float rv[2] = {0.f, 0.f}, rk[2] = {0.f, 0.f};
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = r0 + (lane >> 2) + 8 * hr;
      const float bi = sm.bet[i];
      const size_t off = ((size_t)(t0 + i) * p.nh + h) * kD + d0;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int j = 8 * n + 2 * (lane & 3);
        const float2 vv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.V[i * kS128 + d0 + j]));
        const float2 kb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.KB[i * kS128 + d0 + j]));
        rv[hr] += cv[n][2 * hr] * vv.x + cv[n][2 * hr + 1] * vv.y;
        rk[hr] += ck[n][2 * hr] * kb.x + ck[n][2 * hr + 1] * kb.y;
        if (i < len) {
          *reinterpret_cast<uint32_t*>(p.dv + off + j) = pack2(bi * cv[n][2 * hr], bi * cv[n][2 * hr + 1]);
          const float e0 = __expf(sm.G[i * kG + d0 + j]), e1 = __expf(sm.G[i * kG + d0 + j + 1]);
          float2 ka = kav[hr][n];
          ka.x += bi * ck[n][2 * hr] * e0;
          ka.y += bi * ck[n][2 * hr + 1] * e1;
          *reinterpret_cast<float2*>(p.dKa + off + j) = ka;
          float2 ga = gav[hr][n];
          ga.x += bi * ck[n][2 * hr] * kb.x;
          ga.y += bi * ck[n][2 * hr + 1] * kb.y;
          *reinterpret_cast<float2*>(p.dgam + off + j) = ga;
        }
      }
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = r0 + (lane >> 2) + 8 * hr;
      const float v_ = quad_sum(rv[hr]), k_ = quad_sum(rk[hr]);
      if ((lane & 3) == 0) sm.pb[warp >> 2][i] = v_ + k_;
    }
  }
  __syncthreads();
  if (tid < len)
    p.dbeta[(size_t)(t0 + tid) * p.nh + h] =
        sm.dbs[tid] + (((sm.pb[0][tid] + sm.pb[1][tid]) + sm.pb[2][tid]) + sm.pb[3][tid]);
}

// ============================================================== Kimi Delta backward: the per-channel decay terms
// The gradients that pass through e^(gamma_ic - gamma_jc) inside the masked
// q.k block (N = its gradient) and A (M = diag(beta) dA):
//     a_ic = sum_{j<=i} N_ij k_jc E_ijc     m_ic = sum_{j<i} M_ij k_jc E_ijc
//     b_jc = sum_{i>=j} N_ij q_ic E_ijc     n_jc = sum_{i>j} M_ij k_ic E_ijc,
// E_ijc = e^(gamma_ic - gamma_jc); then the final dq = dQa + a,
// dk = dKa + b + m + n, dgam += q o a - k o b + k o m - k o n and
// dg = reverse running sum of dgam over the chunk.  The exponent is split at
// the first row r of i's 16-row block I, as in the forward's prep:
//     a_I = e^(gamma_I - gamma_r) o (N_I. KI_I),   KI_I = K_j o e^(gamma_r - gamma_j)
//     b_J = sum_{I >= J} e^(gamma_r - gamma_J) o (N_IJ^T (Q_I o e^(gamma_I - gamma_r)))
// (and m, n with M and K), so every sum is a matrix product.  Warp w owns rows
// [16 (w % 4), +16) x channels [32 (w / 4), +32) of a, m, b and n.
struct KdaExpSmem {
  __nv_bfloat16 N[kC * kS64];
  __nv_bfloat16 M[kC * kS64];
  __nv_bfloat16 K[kC * kS128];
  __nv_bfloat16 Q[kC * kS128];
  __nv_bfloat16 KBr[kC * kS128];   // K o e^(gamma - gamma_r)
  __nv_bfloat16 QBr[kC * kS128];   // Q o e^(gamma - gamma_r)
  __nv_bfloat16 KI[160 * kS128];   // per row block I: K_j o e^(gamma_rI - gamma_j), j < 16 (I + 1)
  float G[kC * kG];                // gamma per channel, then dgam
  float tot[4 * kD];               // scratch of the channel running sums
};
static_assert(sizeof(KdaExpSmem) <= 227 * 1024, "fits one SM");

__global__ void __launch_bounds__(kLocalThreads) kda_bwd_exp_kernel(GdnParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  KdaExpSmem& sm = *reinterpret_cast<KdaExpSmem*>(smem_raw);
  constexpr int nt = kLocalThreads;
  grid_dependency_wait();
  const int ci = blockIdx.x, h = blockIdx.y;
  const int n_chunks = __ldcg(p.hdr);
  const int4 ch = p.chunks[ci];
  if (ci >= n_chunks) return;
  const int len = chunk_len(ch, p.total);
  if (len <= 0) return;  // only with a boundary list that breaks its rules
  const int t0 = ch.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sN = smem_u32(sm.N), sM = smem_u32(sm.M), sKBr = smem_u32(sm.KBr), sQBr = smem_u32(sm.QBr),
                 sKI = smem_u32(sm.KI);
  load_rows128(smem_u32(sm.K), p.k, t0, len, h, p.nh, tid, nt);
  load_rows128(smem_u32(sm.Q), p.q, t0, len, h, p.nh, tid, nt);
  for (int e = tid; e < kC * 32; e += nt) {
    const int r = e >> 5, cc = (e & 31) * 4;
    const bool ok = r < len;
    cp_async16(smem_u32(&sm.G[r * kG + cc]), p.g + ((size_t)(t0 + (ok ? r : 0)) * p.nh + h) * kD + cc, ok);
  }
  cp_async_commit();
  {
    const size_t base = ((size_t)ci * p.nh + h) * (kC * kC);
    constexpr int kRounds = kC * kC / 2 / nt;
    static_assert(kC * kC / 2 % nt == 0, "whole rounds");
    float2 nv[kRounds], mv[kRounds];  // all loads in flight before the first store
#pragma unroll
    for (int k = 0; k < kRounds; ++k) {
      const int e = tid + k * nt;
      nv[k] = *reinterpret_cast<const float2*>(p.Nw + base + 2 * e);
      mv[k] = *reinterpret_cast<const float2*>(p.Mw + base + 2 * e);
    }
#pragma unroll
    for (int k = 0; k < kRounds; ++k) {
      const int e = tid + k * nt, i = e >> 5, j = (e & 31) * 2;
      *reinterpret_cast<uint32_t*>(&sm.N[i * kS64 + j]) = pack2(nv[k].x, nv[k].y);
      *reinterpret_cast<uint32_t*>(&sm.M[i * kS64 + j]) = pack2(mv[k].x, mv[k].y);
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  chan_running_sum(sm.G, sm.tot, tid);  // gamma per channel
  for (int e = tid; e < kC * kD / 8; e += nt) {  // eight channels per thread
    const int i = e >> 4, q = e & 15;
    const int r = i & ~15;
    scale_row8(&sm.KBr[i * kS128], &sm.K[i * kS128], &sm.G[i * kG], &sm.G[r * kG], q);
    scale_row8(&sm.QBr[i * kS128], &sm.Q[i * kS128], &sm.G[i * kG], &sm.G[r * kG], q);
  }
  for (int e = tid; e < 160 * kD / 8; e += nt) {
    const int row = e >> 4, q = e & 15;
    const int I = row < 16 ? 0 : (row < 48 ? 1 : (row < 96 ? 2 : 3));
    const int j = row - ki_row0(I), r = 16 * I;
    scale_row8(&sm.KI[row * kS128], &sm.K[j * kS128], &sm.G[r * kG], &sm.G[j * kG], q);
  }
  __syncthreads();
  const int R = warp & 3, r0 = 16 * R, c0 = 32 * (warp >> 2);
  float pa[4][4], pm[4][4], pb[4][4], pn[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) pa[n][e] = pm[n][e] = pb[n][e] = pn[n][e] = 0.f;
  // a, m: rows of block R against KI_R (columns j < 16 (R + 1))
  for (int J = 0; J <= R; ++J) {
    uint32_t an[4], am[4];
    ldsm_x4(an, frag_a(sN, kS64, r0, 16 * J, lane));
    ldsm_x4(am, frag_a(sM, kS64, r0, 16 * J, lane));
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t b[4];
      ldsm_x4_t(b, frag_b(sKI, kS128, ki_row0(R) + 16 * J, c0 + 16 * np, lane));
      mma_bf16(pa[2 * np], an, b[0], b[1]);
      mma_bf16(pa[2 * np + 1], an, b[2], b[3]);
      mma_bf16(pm[2 * np], am, b[0], b[1]);
      mma_bf16(pm[2 * np + 1], am, b[2], b[3]);
    }
  }
  // b, n: columns j of block R, from every row block I >= R, each with its own reference
  for (int I = R; I < 4; ++I) {
    float tb[4][4], tn[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) tb[n][e] = tn[n][e] = 0.f;
    uint32_t an[4], am[4];
    ldsm_x4_t(an, frag_bt(sN, kS64, 16 * I, r0, lane));  // N_IR^T: N stored [i][j]
    ldsm_x4_t(am, frag_bt(sM, kS64, 16 * I, r0, lane));
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t bq[4], bk[4];
      ldsm_x4_t(bq, frag_b(sQBr, kS128, 16 * I, c0 + 16 * np, lane));
      ldsm_x4_t(bk, frag_b(sKBr, kS128, 16 * I, c0 + 16 * np, lane));
      mma_bf16(tb[2 * np], an, bq[0], bq[1]);
      mma_bf16(tb[2 * np + 1], an, bq[2], bq[3]);
      mma_bf16(tn[2 * np], am, bk[0], bk[1]);
      mma_bf16(tn[2 * np + 1], am, bk[2], bk[3]);
    }
    const int rI = 16 * I;
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = r0 + (lane >> 2) + 8 * (e >> 1);
        const int cc = c0 + 8 * n + 2 * (lane & 3) + (e & 1);
        const float f = __expf(sm.G[rI * kG + cc] - sm.G[j * kG + cc]);
        pb[n][e] = fmaf(f, tb[n][e], pb[n][e]);
        pn[n][e] = fmaf(f, tn[n][e], pn[n][e]);
      }
  }
  // epilogue: this thread's (row, channel) elements, two adjacent channels at
  // a time.  The fp32 partial gradients of channel group n + 1 are read
  // before group n's stores, so each group's reads overlap the previous
  // group's work (rows past the chunk read row 0 instead, never used).
  float dgv[4][4];
  float2 nxt[3][2];
  auto read_group = [&](float2 (&v)[3][2], int n) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = r0 + (lane >> 2) + 8 * hr;
      const size_t off = ((size_t)(t0 + (i < len ? i : 0)) * p.nh + h) * kD + c0 + 8 * n + 2 * (lane & 3);
      v[0][hr] = *reinterpret_cast<const float2*>(p.dQa + off);
      v[1][hr] = *reinterpret_cast<const float2*>(p.dKa + off);
      v[2][hr] = *reinterpret_cast<const float2*>(p.dgam + off);
    }
  };
  read_group(nxt, 0);
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    float2 qav[2], kav[2], gav[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) qav[hr] = nxt[0][hr], kav[hr] = nxt[1][hr], gav[hr] = nxt[2][hr];
    if (n + 1 < 4) read_group(nxt, n + 1);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = r0 + (lane >> 2) + 8 * hr;
      const int cc = c0 + 8 * n + 2 * (lane & 3);
      float a[2], m[2], b[2], nn[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float f = __expf(sm.G[i * kG + cc + u] - sm.G[r0 * kG + cc + u]);
        a[u] = f * pa[n][2 * hr + u];
        m[u] = f * pm[n][2 * hr + u];
        b[u] = pb[n][2 * hr + u];
        nn[u] = pn[n][2 * hr + u];
      }
      const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.K[i * kS128 + cc]));
      const float2 qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.Q[i * kS128 + cc]));
      float dg0 = 0.f, dg1 = 0.f;
      if (i < len) {
        const size_t off = ((size_t)(t0 + i) * p.nh + h) * kD + cc;
        const float2 qa = qav[hr], ka = kav[hr], ga = gav[hr];
        *reinterpret_cast<uint32_t*>(p.dq + off) = pack2(qa.x + a[0], qa.y + a[1]);
        *reinterpret_cast<uint32_t*>(p.dk + off) = pack2(ka.x + b[0] + m[0] + nn[0], ka.y + b[1] + m[1] + nn[1]);
        dg0 = ga.x + qv.x * a[0] + kv.x * (m[0] - b[0] - nn[0]);
        dg1 = ga.y + qv.y * a[1] + kv.y * (m[1] - b[1] - nn[1]);
      }
      dgv[n][2 * hr] = dg0;
      dgv[n][2 * hr + 1] = dg1;
    }
  }
  __syncthreads();  // gamma no longer read: dgam goes in its place
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      sm.G[(r0 + (lane >> 2) + 8 * (e >> 1)) * kG + c0 + 8 * n + 2 * (lane & 3) + (e & 1)] = dgv[n][e];
  __syncthreads();
  // dg = reverse running sum of dgam down each channel: four 16-row
  // segments at once, each adding the totals of the segments below it
  {
    const int c = tid & (kD - 1), sg = tid >> 7, i0 = 16 * sg;
    float acc = 0.f;
    for (int i = i0 + 15; i >= i0; --i) acc += sm.G[i * kG + c];
    sm.tot[sg * kD + c] = acc;
    __syncthreads();
    float off = 0.f;
    for (int s2 = 3; s2 > sg; --s2) off += sm.tot[s2 * kD + c];
    acc = off;
    for (int i = i0 + 15; i >= i0; --i) {
      acc += sm.G[i * kG + c];
      if (i < len) p.dg[((size_t)(t0 + i) * p.nh + h) * kD + c] = acc;
    }
  }
}

}  // namespace

// Workspace layout: offsets off[0..6] of the forward's regions (header,
// chunk table, segment table, W, U, Aqk, gamma); with bwd, off[7..13] of the
// backward's (H0, dH1, E, dE, dW, dKa, dgam); with kda (a decay per channel),
// off[14..16] (QB, KC, e^gamma_last), and with both off[17..22] (X, A
// unscaled, N, M, dQa, dgam per channel).  Returns the total size.
size_t gdn_workspace_layout(int64_t total, int nh, int nseg, size_t off[23], bool bwd, bool kda = false) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t max_chunks = (size_t)(total / kC) + (size_t)nseg + 1;
  const size_t tok = (size_t)total * nh * kD;  // elements of a [T, H, 128] tensor
  const size_t states = max_chunks * nh * kD * kD;
  size_t o = 0;
  off[0] = o; o += 256;                                      // header
  off[1] = o; o += up(max_chunks * sizeof(int4));            // chunk table
  off[2] = o; o += up((size_t)nseg * sizeof(int4) + 16);     // segment table
  off[3] = o; o += up(tok * 2);                              // W
  off[4] = o; o += up(tok * 2);                              // U
  off[5] = o; o += up(max_chunks * nh * kC * kC * 2);        // Aqk
  off[6] = o; o += up((size_t)total * nh * sizeof(float));   // gamma
  if (bwd) {
    off[7] = o; o += up(states * 2);                         // H0
    off[8] = o; o += up(states * 2);                         // dH1
    off[9] = o; o += up(tok * 2);                            // E
    off[10] = o; o += up(tok * 2);                           // dE
    off[11] = o; o += up(tok * 2);                           // dW
    off[12] = o; o += up(tok * 4);                           // dKa
    off[13] = o; o += up((size_t)total * nh * sizeof(float)); // dgam
  }
  if (kda) {
    off[14] = o; o += up(tok * 2);                           // QB
    off[15] = o; o += up(tok * 2);                           // KC
    off[16] = o; o += up(max_chunks * nh * kD * sizeof(float)); // e^gamma_last per chunk and channel
    if (bwd) {
      const size_t blk = up(max_chunks * nh * kC * kC * sizeof(float));
      off[17] = o; o += blk;                                 // X
      off[18] = o; o += blk;                                 // A unscaled
      off[19] = o; o += blk;                                 // N
      off[20] = o; o += blk;                                 // M
      off[21] = o; o += up(tok * 4);                         // dQa
      off[22] = o; o += up(tok * 4);                         // dgam per channel
    }
  }
  return o;
}

// Argument checks shared by the forward and the backward, then the parameter
// block over the workspace.  Returns an ATTN_* code.
int gdn_setup(GdnParams& p, const void* q, const void* k, const void* v, const float* g, const float* beta,
              const int32_t* cu_seqlens, float scale, void* workspace, size_t workspace_bytes, int64_t total,
              int32_t num_heads, int32_t head_dim, int32_t num_segments, bool bwd, bool kda = false) {
  if (!q || !k || !v || !g || !beta || !cu_seqlens || !workspace) return ATTN_ERR_NULL_POINTER;
  if (total < 0 || num_heads <= 0 || num_segments < 0 || (num_segments == 0 && total > 0)) return ATTN_ERR_SHAPE;
  if (head_dim != kD) return ATTN_ERR_HEAD_DIM;
  if (total > (1LL << 30) || num_heads > 1024 || (long long)num_segments > (1LL << 24) ||
      total * num_heads > (1LL << 31) || (long long)num_segments * num_heads * (kD / kDvb) >= (1LL << 31))
    return ATTN_ERR_TOO_LARGE;
  if (!std::isfinite(scale)) return ATTN_ERR_SCALE;
  const void* ptrs[] = {q, k, v, g, beta, cu_seqlens};
  for (const void* x : ptrs)
    if (reinterpret_cast<uintptr_t>(x) & 15u) return ATTN_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_ALIGNMENT;
  size_t off[23];
  if (workspace_bytes < gdn_workspace_layout(total, num_heads, num_segments, off, bwd, kda)) return ATTN_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p = GdnParams{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.g = g;
  p.beta = beta;
  p.cu = cu_seqlens;
  p.total = (int)total;
  p.nh = num_heads;
  p.nseg = num_segments;
  p.max_chunks = (int)(total / kC) + num_segments + 1;
  p.scale = scale;
  p.hdr = reinterpret_cast<int*>(ws + off[0]);
  p.chunks = reinterpret_cast<int4*>(ws + off[1]);
  p.segs = reinterpret_cast<int4*>(ws + off[2]);
  p.W = reinterpret_cast<__nv_bfloat16*>(ws + off[3]);
  p.U = reinterpret_cast<__nv_bfloat16*>(ws + off[4]);
  p.Aqk = reinterpret_cast<__nv_bfloat16*>(ws + off[5]);
  p.gam = reinterpret_cast<float*>(ws + off[6]);
  if (bwd) {
    p.H0 = reinterpret_cast<__nv_bfloat16*>(ws + off[7]);
    p.dH1 = reinterpret_cast<__nv_bfloat16*>(ws + off[8]);
    p.E = reinterpret_cast<__nv_bfloat16*>(ws + off[9]);
    p.dE = reinterpret_cast<__nv_bfloat16*>(ws + off[10]);
    p.dW = reinterpret_cast<__nv_bfloat16*>(ws + off[11]);
    p.dKa = reinterpret_cast<float*>(ws + off[12]);
    p.dgam = reinterpret_cast<float*>(ws + off[13]);
  }
  if (kda) {
    p.QB = reinterpret_cast<__nv_bfloat16*>(ws + off[14]);
    p.KC = reinterpret_cast<__nv_bfloat16*>(ws + off[15]);
    p.Bc = reinterpret_cast<float*>(ws + off[16]);
    if (bwd) {
      p.Xw = reinterpret_cast<float*>(ws + off[17]);
      p.Araw = reinterpret_cast<float*>(ws + off[18]);
      p.Nw = reinterpret_cast<float*>(ws + off[19]);
      p.Mw = reinterpret_cast<float*>(ws + off[20]);
      p.dQa = reinterpret_cast<float*>(ws + off[21]);
      p.dgam = reinterpret_cast<float*>(ws + off[22]);
    }
  }
  return ATTN_OK;
}

// The planner and the per-chunk WY factors, shared by both directions.
cudaError_t launch_gdn_prep(const GdnParams& p, cudaStream_t s) {
  cudaError_t e = launch_pdl(gdn_plan_kernel, dim3(1), dim3(256), 0, s, p);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gdn_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(PrepSmem));
  if (e == cudaSuccess)
    e = launch_pdl(gdn_prep_kernel, dim3((unsigned)p.max_chunks, (unsigned)p.nh), dim3(kGdnThreads),
                   sizeof(PrepSmem), s, p);
  return e;
}

// The planner and the per-chunk factors with a decay per channel.
cudaError_t launch_kda_prep(const GdnParams& p, cudaStream_t s) {
  cudaError_t e = launch_pdl(gdn_plan_kernel, dim3(1), dim3(256), 0, s, p);
  auto kern = p.Xw ? kda_prep_kernel<true> : kda_prep_kernel<false>;
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(KdaPrepSmem));
  if (e == cudaSuccess)
    e = launch_pdl(kern, dim3((unsigned)p.max_chunks, (unsigned)p.nh), dim3(kLocalThreads), sizeof(KdaPrepSmem), s,
                   p);
  return e;
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess && f)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// An N-D bf16 map: sizes (innermost first), byte strides of the outer
// dimensions, box, swizzle.  Out-of-range rows read as zero.
template <int N>
bool encode_bf16_map(CUtensorMap* m, const void* base, const cuuint64_t (&dims)[N],
                     const cuuint64_t (&strides)[N - 1], const cuuint32_t (&box)[N],
                     CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint32_t es[N];
  for (int i = 0; i < N; ++i) es[i] = 1;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The state passes' maps (StateMaps) over the inputs and the workspace.
int make_state_maps(StateMaps& m, const GdnParams& p) {
  // (64 columns, token, column half, head): the box's order in shared memory
  // is [half][token][64 columns], the two swizzled halves of the tile
  const cuuint64_t rows[4] = {64, (cuuint64_t)p.total, 2, (cuuint64_t)p.nh};
  const cuuint64_t row_str[3] = {(cuuint64_t)p.nh * kD * 2, 64 * 2, (cuuint64_t)kD * 2};
  const cuuint32_t row_box[4] = {64, (cuuint32_t)kC, 2, 1};
  const cuuint64_t blocks[3] = {(cuuint64_t)kC, (cuuint64_t)kC, (cuuint64_t)p.max_chunks * p.nh};
  const cuuint64_t blk_str[2] = {(cuuint64_t)kC * 2, (cuuint64_t)kC * kC * 2};
  const cuuint32_t blk_box[3] = {(cuuint32_t)kC, (cuuint32_t)kC, 1};
  // value columns: (128 columns, head, token), box 32 columns x 1 x 64 tokens
  const cuuint64_t cols[3] = {(cuuint64_t)kD, (cuuint64_t)p.nh, (cuuint64_t)p.total};
  const cuuint64_t col_str[2] = {(cuuint64_t)kD * 2, (cuuint64_t)p.nh * kD * 2};
  const cuuint32_t col_box[3] = {(cuuint32_t)kDvb, 1, (cuuint32_t)kC};
  const bool chan = p.KC != nullptr;  // Kimi Delta
  m = StateMaps{};
  bool ok = encode_bf16_map(&m.w, p.W, rows, row_str, row_box) &&
            encode_bf16_map(&m.k, chan ? p.KC : p.k, rows, row_str, row_box) &&
            encode_bf16_map(&m.q, chan ? p.QB : p.q, rows, row_str, row_box) &&
            encode_bf16_map(&m.aq, p.Aqk, blocks, blk_str, blk_box) &&
            encode_bf16_map(&m.u, p.U, cols, col_str, col_box, CU_TENSOR_MAP_SWIZZLE_64B);
  if (ok && p.dO) ok = encode_bf16_map(&m.d_o, p.dO, cols, col_str, col_box, CU_TENSOR_MAP_SWIZZLE_64B);
  return ok ? ATTN_OK : ATTN_ERR_CUDA;
}

// A state pass: the maps, the parameters, and 1024 bytes of shared-memory
// slack for the stage alignment.
template <typename Smem, typename... KArgs>
cudaError_t launch_state(void (*kernel)(KArgs...), dim3 grid, cudaStream_t s, const StateMaps& m,
                         const GdnParams& p) {
  const int bytes = (int)sizeof(Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) e = launch_pdl(kernel, grid, dim3(kStateBlock), (size_t)bytes, s, m, p);
  return e;
}

template <typename Smem, typename... KArgs>
cudaError_t launch_big(void (*kernel)(KArgs...), dim3 grid, cudaStream_t s, const GdnParams& p,
                       int threads = kStateThreads) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
  if (e == cudaSuccess) e = launch_pdl(kernel, grid, dim3(threads), sizeof(Smem), s, p);
  return e;
}

// The forward's checks and set-up.  `save`: the workspace is the backward's
// (the saving forward keeps what the backward would recompute there).
int fwd_entry(GdnParams& p, StateMaps& maps, const void* q, const void* k, const void* v, const float* g,
              const float* beta, const int32_t* cu_seqlens, float scale, void* o, void* workspace,
              size_t workspace_bytes, int64_t total, int32_t num_heads, int32_t head_dim, int32_t num_segments,
              bool kda, bool save) {
  int rc = gdn_setup(p, q, k, v, g, beta, cu_seqlens, scale, workspace, workspace_bytes, total, num_heads, head_dim,
                     num_segments, save, kda);
  if (rc) return rc;
  if (!o) return ATTN_ERR_NULL_POINTER;
  if (reinterpret_cast<uintptr_t>(o) & 15u) return ATTN_ERR_ALIGNMENT;
  int* status = nullptr;
  int sms = 0;
  if ((rc = device_for_call(&status, &sms))) return rc;
  if (total == 0) return ATTN_OK;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.status = status;
  return make_state_maps(maps, p);
}

// The backward's checks and set-up.
int bwd_entry(GdnParams& p, StateMaps& maps, const void* q, const void* k, const void* v, const float* g,
              const float* beta, const void* d_o, const int32_t* cu_seqlens, float scale, void* dq, void* dk,
              void* dv, float* dg, float* dbeta, void* workspace, size_t workspace_bytes, int64_t total,
              int32_t num_heads, int32_t head_dim, int32_t num_segments, bool kda) {
  int rc = gdn_setup(p, q, k, v, g, beta, cu_seqlens, scale, workspace, workspace_bytes, total, num_heads, head_dim,
                     num_segments, true, kda);
  if (rc) return rc;
  const void* outs[] = {d_o, dq, dk, dv, dg, dbeta};
  for (const void* x : outs)
    if (!x) return ATTN_ERR_NULL_POINTER;
  for (const void* x : outs)
    if (reinterpret_cast<uintptr_t>(x) & 15u) return ATTN_ERR_ALIGNMENT;
  int* status = nullptr;
  int sms = 0;
  if ((rc = device_for_call(&status, &sms))) return rc;
  if (total == 0) return ATTN_OK;
  p.dO = static_cast<const __nv_bfloat16*>(d_o);
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.dg = dg;
  p.dbeta = dbeta;
  p.status = status;
  return make_state_maps(maps, p);
}

dim3 seg_grid_of(const GdnParams& p) { return dim3((unsigned)((long long)p.nseg * p.nh * (kD / kDvb))); }
dim3 chunk_grid_of(const GdnParams& p) { return dim3((unsigned)p.max_chunks, (unsigned)p.nh); }

// The forward.  save: O and, for the backward, the chunk-start states and E.
cudaError_t launch_layer_fwd(const GdnParams& p, const StateMaps& maps, cudaStream_t s, bool kda, bool save) {
  cudaError_t e = kda ? launch_kda_prep(p, s) : launch_gdn_prep(p, s);
  if (e != cudaSuccess) return e;
  if (kda)
    return save ? launch_state<StateSmem>(gdn_state_kernel<true, true, true>, seg_grid_of(p), s, maps, p)
                : launch_state<StateSmem>(gdn_state_kernel<true, false, true>, seg_grid_of(p), s, maps, p);
  return save ? launch_state<StateSmem>(gdn_state_kernel<true, true, false>, seg_grid_of(p), s, maps, p)
              : launch_state<StateSmem>(gdn_state_kernel<true, false, false>, seg_grid_of(p), s, maps, p);
}

// The backward.  saved: the workspace already holds the saving forward's
// factors, states and E, so the plan, the prep and the recomputation are skipped.
cudaError_t launch_layer_bwd(const GdnParams& p, const StateMaps& maps, cudaStream_t s, bool kda, bool saved) {
  const dim3 seg_grid = seg_grid_of(p), chunk_grid = chunk_grid_of(p);
  cudaError_t e = cudaSuccess;
  if (!saved) {
    e = kda ? launch_kda_prep(p, s) : launch_gdn_prep(p, s);
    if (e == cudaSuccess)
      e = kda ? launch_state<StateSmem>(gdn_state_kernel<false, true, true>, seg_grid, s, maps, p)
              : launch_state<StateSmem>(gdn_state_kernel<false, true, false>, seg_grid, s, maps, p);
  }
  if (kda) {
    if (e == cudaSuccess) e = launch_state<BwdStateSmem>(gdn_bwd_state_kernel<true>, seg_grid, s, maps, p);
    if (e == cudaSuccess) e = launch_big<KdaLocalHSmem>(kda_bwd_local_h_kernel, chunk_grid, s, p, kLocalThreads);
    if (e == cudaSuccess) e = launch_big<KdaLocalWySmem>(kda_bwd_local_wy_kernel, chunk_grid, s, p, kLocalThreads);
    if (e == cudaSuccess) e = launch_big<KdaExpSmem>(kda_bwd_exp_kernel, chunk_grid, s, p, kLocalThreads);
  } else {
    if (e == cudaSuccess) e = launch_state<BwdStateSmem>(gdn_bwd_state_kernel<false>, seg_grid, s, maps, p);
    if (e == cudaSuccess) e = launch_big<LocalHSmem>(gdn_bwd_local_h_kernel, chunk_grid, s, p, kLocalThreads);
    if (e == cudaSuccess) e = launch_big<LocalWySmem>(gdn_bwd_local_wy_kernel, chunk_grid, s, p, kLocalThreads);
  }
  return e;
}

int run_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
            const int32_t* cu_seqlens, float scale, void* o, void* workspace, size_t workspace_bytes, int64_t total,
            int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream, bool kda, bool save) {
  GdnParams p;
  StateMaps maps;
  const int rc = fwd_entry(p, maps, q, k, v, g, beta, cu_seqlens, scale, o, workspace, workspace_bytes, total,
                           num_heads, head_dim, num_segments, kda, save);
  if (rc || total == 0) return rc;
  const cudaError_t e = launch_layer_fwd(p, maps, static_cast<cudaStream_t>(stream), kda, save);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int run_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta, const void* d_o,
            const int32_t* cu_seqlens, float scale, void* dq, void* dk, void* dv, float* dg, float* dbeta,
            void* workspace, size_t workspace_bytes, int64_t total, int32_t num_heads, int32_t head_dim,
            int32_t num_segments, void* stream, bool kda, bool saved) {
  GdnParams p;
  StateMaps maps;
  const int rc = bwd_entry(p, maps, q, k, v, g, beta, d_o, cu_seqlens, scale, dq, dk, dv, dg, dbeta, workspace,
                           workspace_bytes, total, num_heads, head_dim, num_segments, kda);
  if (rc || total == 0) return rc;
  const cudaError_t e = launch_layer_bwd(p, maps, static_cast<cudaStream_t>(stream), kda, saved);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace vsw

extern "C" {

size_t gdn_varlen_workspace_bytes(int64_t total, int32_t num_heads, int32_t num_segments) {
  if (total < 0 || num_heads <= 0 || num_segments < 0 || total > (1LL << 30) || num_heads > 1024) return 0;
  size_t off[23];
  return vsw::gdn_workspace_layout(total, num_heads, num_segments, off, false);
}

size_t gdn_varlen_bwd_workspace_bytes(int64_t total, int32_t num_heads, int32_t num_segments) {
  if (total < 0 || num_heads <= 0 || num_segments < 0 || total > (1LL << 30) || num_heads > 1024) return 0;
  size_t off[23];
  return vsw::gdn_workspace_layout(total, num_heads, num_segments, off, true);
}

int gdn_varlen_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                   const int32_t* cu_seqlens, float scale, void* o, void* workspace, size_t workspace_bytes,
                   int64_t total, int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream) {
  return vsw::run_fwd(q, k, v, g, beta, cu_seqlens, scale, o, workspace, workspace_bytes, total, num_heads, head_dim,
                      num_segments, stream, false, false);
}

int gdn_varlen_fwd_save(const void* q, const void* k, const void* v, const float* g, const float* beta,
                        const int32_t* cu_seqlens, float scale, void* o, void* workspace, size_t workspace_bytes,
                        int64_t total, int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream) {
  return vsw::run_fwd(q, k, v, g, beta, cu_seqlens, scale, o, workspace, workspace_bytes, total, num_heads, head_dim,
                      num_segments, stream, false, true);
}

int gdn_varlen_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta, const void* d_o,
                   const int32_t* cu_seqlens, float scale, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                   void* workspace, size_t workspace_bytes, int64_t total, int32_t num_heads, int32_t head_dim,
                   int32_t num_segments, void* stream) {
  return vsw::run_bwd(q, k, v, g, beta, d_o, cu_seqlens, scale, dq, dk, dv, dg, dbeta, workspace, workspace_bytes,
                      total, num_heads, head_dim, num_segments, stream, false, false);
}

int gdn_varlen_bwd_saved(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const void* d_o, const int32_t* cu_seqlens, float scale, void* dq, void* dk, void* dv,
                         float* dg, float* dbeta, void* workspace, size_t workspace_bytes, int64_t total,
                         int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream) {
  return vsw::run_bwd(q, k, v, g, beta, d_o, cu_seqlens, scale, dq, dk, dv, dg, dbeta, workspace, workspace_bytes,
                      total, num_heads, head_dim, num_segments, stream, false, true);
}

size_t kda_varlen_workspace_bytes(int64_t total, int32_t num_heads, int32_t num_segments) {
  if (total < 0 || num_heads <= 0 || num_segments < 0 || total > (1LL << 30) || num_heads > 1024) return 0;
  size_t off[23];
  return vsw::gdn_workspace_layout(total, num_heads, num_segments, off, false, true);
}

size_t kda_varlen_bwd_workspace_bytes(int64_t total, int32_t num_heads, int32_t num_segments) {
  if (total < 0 || num_heads <= 0 || num_segments < 0 || total > (1LL << 30) || num_heads > 1024) return 0;
  size_t off[23];
  return vsw::gdn_workspace_layout(total, num_heads, num_segments, off, true, true);
}

int kda_varlen_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                   const int32_t* cu_seqlens, float scale, void* o, void* workspace, size_t workspace_bytes,
                   int64_t total, int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream) {
  return vsw::run_fwd(q, k, v, g, beta, cu_seqlens, scale, o, workspace, workspace_bytes, total, num_heads, head_dim,
                      num_segments, stream, true, false);
}

int kda_varlen_fwd_save(const void* q, const void* k, const void* v, const float* g, const float* beta,
                        const int32_t* cu_seqlens, float scale, void* o, void* workspace, size_t workspace_bytes,
                        int64_t total, int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream) {
  return vsw::run_fwd(q, k, v, g, beta, cu_seqlens, scale, o, workspace, workspace_bytes, total, num_heads, head_dim,
                      num_segments, stream, true, true);
}

int kda_varlen_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta, const void* d_o,
                   const int32_t* cu_seqlens, float scale, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                   void* workspace, size_t workspace_bytes, int64_t total, int32_t num_heads, int32_t head_dim,
                   int32_t num_segments, void* stream) {
  return vsw::run_bwd(q, k, v, g, beta, d_o, cu_seqlens, scale, dq, dk, dv, dg, dbeta, workspace, workspace_bytes,
                      total, num_heads, head_dim, num_segments, stream, true, false);
}

int kda_varlen_bwd_saved(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const void* d_o, const int32_t* cu_seqlens, float scale, void* dq, void* dk, void* dv,
                         float* dg, float* dbeta, void* workspace, size_t workspace_bytes, int64_t total,
                         int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream) {
  return vsw::run_bwd(q, k, v, g, beta, d_o, cu_seqlens, scale, dq, dk, dv, dg, dbeta, workspace, workspace_bytes,
                      total, num_heads, head_dim, num_segments, stream, true, true);
}

}  // extern "C"
