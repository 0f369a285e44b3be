// Gated DeltaNet forward over packed documents (gdn_varlen.h).
//
// The recurrence (per head, state H of d_k x d_v = 128 x 128, reset at every
// segment start):
//     e_t = beta_t (v_t - alpha_t H_{t-1}^T k_t),  H_t = alpha_t H_{t-1} + k_t e_t^T,
//     o_t = scale H_t^T q_t,  alpha_t = exp(g_t).
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
// Three kernels:
//   gdn_plan_kernel    one CTA: the chunk table (start, length of every
//                      chunk) and the non-empty segments ordered longest first
//   gdn_prep_kernel    one CTA per (chunk, head), all in parallel: A, Tm,
//                      W, U and the masked Q K^T o Gamma, written to the
//                      workspace (bf16), and gamma (fp32)
//   gdn_state_kernel   one CTA (8 warps) per (segment, head, 32 value
//                      columns): carries H (fp32, in registers) across the
//                      segment's chunks and writes O; the tiles of chunks
//                      c+1 and c+2 load (cp.async) while chunk c computes
// The products are small (64-row) and run in bf16 on the warp-level tensor
// core instruction (mma.sync m16n8k16, fp32 accumulation): the state pass is
// a dependent chain of 64-row steps whose state lives in registers, where the
// asynchronous 128-row tcgen05 path has nothing to overlap.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "attn_internal.h"
#include "attn_varlen.h"
#include "gdn_varlen.h"
#include "ptx.cuh"

namespace vsw {

namespace {

constexpr int kC = 64;         // chunk length (tokens)
constexpr int kD = 128;        // d_k = d_v
constexpr int kDvb = 32;       // value columns per state CTA
constexpr int kGdnThreads = 256;   // prep CTA
constexpr int kStateThreads = 256; // state CTA
constexpr int kS128 = 136;     // smem row stride (elements) of 128-wide bf16 tiles: 272 B, conflict-free ldmatrix
constexpr int kS64 = 72;       // 64-wide: 144 B
constexpr int kS32 = 40;       // 32-wide: 80 B
constexpr int kSF = 65;        // fp32 64 x 64 tiles

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
  // workspace
  int* hdr;             // [0] chunks, [1] non-empty segments
  int4* chunks;         // [max_chunks] {start token, length, segment, chunk index in segment}
  int4* segs;           // [nseg] by length, longest first: {first chunk, chunks, start token, length}
  __nv_bfloat16* W;     // [T, H, 128]
  __nv_bfloat16* U;     // [T, H, 128]
  __nv_bfloat16* Aqk;   // [max_chunks, H, 64, 64]: lower(Q K^T) o Gamma
  float* gam;           // [H, T]: gamma (running log decay within the chunk)
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

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0) : "memory");
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

// ============================================================== prep
// Shared memory of the prep CTA.
struct PrepSmem {
  __nv_bfloat16 K[kC * kS128];
  __nv_bfloat16 Q[kC * kS128];
  __nv_bfloat16 V[kC * kS128];
  float A[kC * kSF];    // A, fp32
  float X[kC * kSF];    // (I + A)^-1, fp32
  float R[3 * 256];     // off-diagonal block products
  __nv_bfloat16 T1[kC * kS64];  // X diag(beta e^gamma)
  __nv_bfloat16 T2[kC * kS64];  // X diag(beta)
  float gam[kC];
  float bet[kC];
};

static_assert(sizeof(PrepSmem) <= 113 * 1024, "two prep CTAs per SM");

__global__ void __launch_bounds__(kGdnThreads, 2) gdn_prep_kernel(GdnParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  PrepSmem& sm = *reinterpret_cast<PrepSmem*>(smem_raw);
  grid_dependency_wait();
  const int c = blockIdx.x, h = blockIdx.y;
  if (c >= p.hdr[0]) return;
  const int4 ch = p.chunks[c];
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
      sm.A[i * kSF + j] = j < i ? bi * G0 * skk[n][2 * hr] : 0.f;
      sm.A[i * kSF + j + 1] = j + 1 < i ? bi * G1 * skk[n][2 * hr + 1] : 0.f;
      *reinterpret_cast<uint32_t*>(aqk + i * kC + j) = pack2(G0 * sqk[n][2 * hr], G1 * sqk[n][2 * hr + 1]);
    }
  }
  __syncthreads();
  // ---- X = (I + A)^-1 (unit lower triangular) in 16 x 16 blocks.
  // Diagonal blocks by forward substitution, one column per thread (threads
  // 64..127 clear the blocks above the diagonal meanwhile):
  //     X_bb[r][c] = [r == c] - sum_{c <= j < r} A_bb[r][j] X_bb[j][c].
  if (tid < 64) {
    const int b = tid >> 4, c = tid & 15, o = 16 * b;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < r; ++j) acc = fmaf(sm.A[(o + r) * kSF + o + j], x[j], acc);
      x[r] = r < c ? 0.f : (r == c ? 1.f : -acc);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) sm.X[(o + r) * kSF + o + c] = x[r];
  } else {
    // blocks (bi, bj) with bi < bj: 6 blocks of 256
    for (int e = tid - 64; e < 6 * 256; e += kGdnThreads - 64) {
      const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
      const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
      const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
      sm.X[(16 * bi + r) * kSF + 16 * bj + c] = 0.f;
    }
  }
  __syncthreads();
  // Blocks below the diagonal, nearest first (d = i - j = 1, 2, 3):
  //     X_ij = -X_ii R_ij,   R_ij = sum_{j <= k < i} A_ik X_kj
  // (the rows of block i of (I + A) X = I).  R goes through sm.R.
  for (int d = 1; d < 4; ++d) {
    const int nb = 4 - d;  // blocks (j + d, j), j = 0 .. nb - 1
    for (int e = tid; e < nb * 256; e += kGdnThreads) {
      const int j = e >> 8, r = (e >> 4) & 15, c = e & 15, i = j + d;
      float acc = 0.f;
      for (int k = 16 * j; k < 16 * i; ++k) acc = fmaf(sm.A[(16 * i + r) * kSF + k], sm.X[k * kSF + 16 * j + c], acc);
      sm.R[e] = acc;
    }
    __syncthreads();
    for (int e = tid; e < nb * 256; e += kGdnThreads) {
      const int j = e >> 8, r = (e >> 4) & 15, c = e & 15, i = j + d;
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) acc = fmaf(sm.X[(16 * i + r) * kSF + 16 * i + k], sm.R[(j << 8) + (k << 4) + c], acc);
      sm.X[(16 * i + r) * kSF + 16 * j + c] = -acc;
    }
    __syncthreads();
  }
  // ---- T1 = X diag(beta e^gamma), T2 = X diag(beta) (bf16)
  for (int e = tid; e < kC * kC / 2; e += kGdnThreads) {
    const int i = e >> 5, j = (e & 31) * 2;
    const float x0 = sm.X[i * kSF + j], x1 = sm.X[i * kSF + j + 1];
    const float b0 = sm.bet[j], b1 = sm.bet[j + 1];
    *reinterpret_cast<uint32_t*>(&sm.T1[i * kS64 + j]) =
        pack2(x0 * b0 * __expf(sm.gam[j]), x1 * b1 * __expf(sm.gam[j + 1]));
    *reinterpret_cast<uint32_t*>(&sm.T2[i * kS64 + j]) = pack2(x0 * b0, x1 * b1);
  }
  __syncthreads();
  // ---- W = T1 K, U = T2 V: warp w rows [16 (w % 4), +16) x columns [64 (w / 4), +64).
  const int d0 = 64 * (warp >> 2);
  float cw[8][4], cu[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) cw[n][e] = cu[n][e] = 0.f;
  const uint32_t sT1 = smem_u32(sm.T1), sT2 = smem_u32(sm.T2);
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

// ============================================================== state + output
struct StateStage {
  __nv_bfloat16 W[kC * kS128];
  __nv_bfloat16 K[kC * kS128];
  __nv_bfloat16 Q[kC * kS128];
  __nv_bfloat16 U[kC * kS32];
  __nv_bfloat16 Aq[kC * kS64];
  float gam[kC];
};
constexpr int kStateStages = 3;  // chunk c + 2 loads while chunk c computes
struct StateSmem {
  StateStage st[kStateStages];
  __nv_bfloat16 H[kD * kS32];   // the state at the chunk start, bf16 (B operand)
  __nv_bfloat16 E[kC * kS32];   // E (bf16)
  __nv_bfloat16 E2[kC * kS32];  // diag(e^(gamma_last - gamma)) E (bf16)
};

static_assert(sizeof(StateSmem) <= 227 * 1024, "the state CTA's shared memory fits one SM");

// Rows of a chunk that lie inside [0, T) (all of them for a valid boundary list).
__device__ __forceinline__ int chunk_len(const int4& ch, int total) {
  return (ch.x < 0 || ch.x >= total) ? 0 : min(ch.y, total - ch.x);
}

__device__ __forceinline__ void load_stage(StateStage& s, const GdnParams& p, int chunk, int h, int vb, int tid) {
  constexpr int nt = kStateThreads;
  const int4 ch = p.chunks[chunk];
  const int len = chunk_len(ch, p.total), t0 = len > 0 ? ch.x : 0;
  load_rows128(smem_u32(s.W), p.W, t0, len, h, p.nh, tid, nt);
  load_rows128(smem_u32(s.K), p.k, t0, len, h, p.nh, tid, nt);
  load_rows128(smem_u32(s.Q), p.q, t0, len, h, p.nh, tid, nt);
  for (int e = tid; e < kC * 4; e += nt) {  // U columns [32 vb, 32 vb + 32)
    const int r = e >> 2, cc = (e & 3) * 8;
    const bool ok = r < len;
    cp_async16(smem_u32(&s.U[r * kS32 + cc]), p.U + ((size_t)(t0 + (ok ? r : 0)) * p.nh + h) * kD + kDvb * vb + cc,
               ok);
  }
  const __nv_bfloat16* aq = p.Aqk + ((size_t)chunk * p.nh + h) * (kC * kC);
  for (int e = tid; e < kC * 8; e += nt) {
    const int r = e >> 3, cc = (e & 7) * 8;
    cp_async16(smem_u32(&s.Aq[r * kS64 + cc]), aq + r * kC + cc, true);
  }
  if (tid < kC) {
    const bool ok = tid < len;
    cp_async4(smem_u32(&s.gam[tid]), p.gam + (size_t)h * p.total + t0 + (ok ? tid : 0), ok);
  }
}

// Eight warps.  Warp w computes, of the chunk's 64 x 32 products (E, Q H,
// O), rows [16 (w % 4), +16) x columns [16 (w / 4), +16), and holds rows
// [16 w, +16) of the 128 x 32 state.
__global__ void __launch_bounds__(kStateThreads) gdn_state_kernel(GdnParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  StateSmem& sm = *reinterpret_cast<StateSmem*>(smem_raw);
  grid_dependency_wait();
  const int per_seg = p.nh * (kD / kDvb);
  const int r = blockIdx.x / per_seg, rem = blockIdx.x - r * per_seg;
  const int h = rem / (kD / kDvb), vb = rem - h * (kD / kDvb);
  if (r >= p.hdr[1]) return;
  const int4 sg = p.segs[r];
  const int first = sg.x, nch = min(sg.y, p.hdr[0] - sg.x);
  if (first < 0 || nch <= 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r0 = 16 * (warp & 3);   // token rows of the E / O products
  const int n0 = 16 * (warp >> 2);  // their value columns
  const int m0 = 16 * warp;         // state rows (d_k)
  float hreg[4][4];                 // state rows [m0, +16) x 32 columns, as mma accumulators (n-tile n)
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) hreg[n][e] = 0.f;
  const uint32_t sH = smem_u32(sm.H), sE = smem_u32(sm.E), sE2 = smem_u32(sm.E2);
  load_stage(sm.st[0], p, first, h, vb, tid);
  cp_async_commit();
  if (nch > 1) load_stage(sm.st[1], p, first + 1, h, vb, tid);
  cp_async_commit();
  for (int ci = 0; ci < nch; ++ci) {
    // Stage (ci + 2) % 3 was last read by chunk ci - 1 (done: the barrier at
    // the end of that chunk).  One group is committed per chunk, so at most
    // the two newest groups (chunks ci + 1, ci + 2) are still in flight.
    if (ci + 2 < nch) load_stage(sm.st[(ci + 2) % kStateStages], p, first + ci + 2, h, vb, tid);
    cp_async_commit();
    cp_async_wait<2>();
    // H (bf16) for this chunk's products
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = m0 + (lane >> 2) + 8 * hr;
        const int j = 8 * n + 2 * (lane & 3);
        *reinterpret_cast<uint32_t*>(&sm.H[i * kS32 + j]) = pack2(hreg[n][2 * hr], hreg[n][2 * hr + 1]);
      }
    __syncthreads();
    StateStage& s = sm.st[ci % kStateStages];
    const int4 ch = p.chunks[first + ci];
    const int t0 = ch.x, len = chunk_len(ch, p.total);
    if (len <= 0) {  // only with a boundary list that breaks its rules
      __syncthreads();
      continue;
    }
    const uint32_t sW = smem_u32(s.W), sK = smem_u32(s.K), sQ = smem_u32(s.Q), sAq = smem_u32(s.Aq);
    const float g_last = s.gam[len - 1];
    // ---- E = U - W H and Q H
    float ce[2][4], cq[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) ce[n][e] = cq[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t aw[4], aq[4], b[4];
      ldsm_x4(aw, frag_a(sW, kS128, r0, 16 * kk, lane));
      ldsm_x4(aq, frag_a(sQ, kS128, r0, 16 * kk, lane));
      ldsm_x4_t(b, frag_b(sH, kS32, 16 * kk, n0, lane));
      mma_bf16(ce[0], aw, b[0], b[1]);
      mma_bf16(ce[1], aw, b[2], b[3]);
      mma_bf16(cq[0], aq, b[0], b[1]);
      mma_bf16(cq[1], aq, b[2], b[3]);
    }
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = r0 + (lane >> 2) + 8 * hr;
        const int j = n0 + 8 * n + 2 * (lane & 3);
        const float2 u = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&s.U[i * kS32 + j]));
        const float e0 = u.x - ce[n][2 * hr], e1 = u.y - ce[n][2 * hr + 1];
        const float w = i < len ? __expf(g_last - s.gam[i]) : 0.f;
        *reinterpret_cast<uint32_t*>(&sm.E[i * kS32 + j]) = pack2(e0, e1);
        *reinterpret_cast<uint32_t*>(&sm.E2[i * kS32 + j]) = pack2(e0 * w, e1 * w);
      }
    __syncthreads();
    // ---- O = scale (e^gamma Q H + Aq E)
    float co[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) co[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) {
      uint32_t a[4], b[4];
      ldsm_x4(a, frag_a(sAq, kS64, r0, 16 * kk, lane));
      ldsm_x4_t(b, frag_b(sE, kS32, 16 * kk, n0, lane));
      mma_bf16(co[0], a, b[0], b[1]);
      mma_bf16(co[1], a, b[2], b[3]);
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = r0 + (lane >> 2) + 8 * hr;
      if (i < len) {
        const float eg = __expf(s.gam[i]);
        __nv_bfloat16* orow = p.o + ((size_t)(t0 + i) * p.nh + h) * kD + kDvb * vb + n0;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          const int j = 8 * n + 2 * (lane & 3);
          *reinterpret_cast<uint32_t*>(orow + j) = pack2(p.scale * (eg * cq[n][2 * hr] + co[n][2 * hr]),
                                                         p.scale * (eg * cq[n][2 * hr + 1] + co[n][2 * hr + 1]));
        }
      }
    }
    // ---- H = e^gamma_last H + K^T E2 (state rows [m0, +16); K^T read from K[token][d_k])
    const float dl = __expf(g_last);
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) hreg[n][e] *= dl;
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) {
      uint32_t a[4], b0[4], b1[4];
      ldsm_x4_t(a, frag_bt(sK, kS128, 16 * kk, m0, lane));
      ldsm_x4_t(b0, frag_b(sE2, kS32, 16 * kk, 0, lane));
      ldsm_x4_t(b1, frag_b(sE2, kS32, 16 * kk, 16, lane));
      mma_bf16(hreg[0], a, b0[0], b0[1]);
      mma_bf16(hreg[1], a, b0[2], b0[3]);
      mma_bf16(hreg[2], a, b1[0], b1[1]);
      mma_bf16(hreg[3], a, b1[2], b1[3]);
    }
    __syncthreads();  // this stage, H, E and E2 are reused by the next chunk
  }
  cp_async_wait<0>();
}

}  // namespace

size_t gdn_workspace_layout(int64_t total, int nh, int nseg, size_t off[7]) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t max_chunks = (size_t)(total / kC) + (size_t)nseg + 1;
  size_t o = 0;
  off[0] = o; o += 256;                                                    // header
  off[1] = o; o += up(max_chunks * sizeof(int4));                          // chunk table
  off[2] = o; o += up((size_t)nseg * sizeof(int4) + 16);                   // segment table
  off[3] = o; o += up((size_t)total * nh * kD * 2);                        // W
  off[4] = o; o += up((size_t)total * nh * kD * 2);                        // U
  off[5] = o; o += up(max_chunks * nh * kC * kC * 2);                      // Aqk
  off[6] = o; o += up((size_t)total * nh * sizeof(float));                 // gamma
  return o;
}

}  // namespace vsw

extern "C" {

size_t gdn_varlen_workspace_bytes(int64_t total, int32_t num_heads, int32_t num_segments) {
  if (total < 0 || num_heads <= 0 || num_segments < 0 || total > (1LL << 30) || num_heads > 1024) return 0;
  size_t off[7];
  return vsw::gdn_workspace_layout(total, num_heads, num_segments, off);
}

int gdn_varlen_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                   const int32_t* cu_seqlens, float scale, void* o, void* workspace, size_t workspace_bytes,
                   int64_t total, int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream) {
  using namespace vsw;
  if (!q || !k || !v || !g || !beta || !cu_seqlens || !o || !workspace) return ATTN_ERR_NULL_POINTER;
  if (total < 0 || num_heads <= 0 || num_segments < 0 || (num_segments == 0 && total > 0)) return ATTN_ERR_SHAPE;
  if (head_dim != kD) return ATTN_ERR_HEAD_DIM;
  if (total > (1LL << 30) || num_heads > 1024 || (long long)num_segments > (1LL << 24) ||
      total * num_heads > (1LL << 31) || (long long)num_segments * num_heads * (kD / kDvb) >= (1LL << 31))
    return ATTN_ERR_TOO_LARGE;
  if (!std::isfinite(scale)) return ATTN_ERR_SCALE;
  const void* ptrs[] = {q, k, v, g, beta, cu_seqlens, o};
  for (const void* x : ptrs)
    if (reinterpret_cast<uintptr_t>(x) & 15u) return ATTN_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_ALIGNMENT;
  size_t off[7];
  if (workspace_bytes < gdn_workspace_layout(total, num_heads, num_segments, off)) return ATTN_ERR_WORKSPACE;
  int* status = nullptr;
  int sms = 0;
  if (int rc = device_for_call(&status, &sms)) return rc;
  if (total == 0) return ATTN_OK;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  GdnParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.g = g;
  p.beta = beta;
  p.cu = cu_seqlens;
  p.o = static_cast<__nv_bfloat16*>(o);
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
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_pdl(gdn_plan_kernel, dim3(1), dim3(256), 0, s, p);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gdn_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(PrepSmem));
  if (e == cudaSuccess)
    e = launch_pdl(gdn_prep_kernel, dim3((unsigned)p.max_chunks, (unsigned)num_heads), dim3(kGdnThreads),
                   sizeof(PrepSmem), s, p);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gdn_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(StateSmem));
  if (e == cudaSuccess)
    e = launch_pdl(gdn_state_kernel, dim3((unsigned)((long long)num_segments * num_heads * (kD / kDvb))),
                   dim3(kStateThreads), sizeof(StateSmem), s, p);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"
