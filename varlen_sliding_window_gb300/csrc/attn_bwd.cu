// Backward pass of document-masked causal grouped-query attention on sm_103a.
//
// With P_ij = exp(s_ij - lse_i), dP_ij = <dout_i, v_j>, D_i = rowsum(dout*out)_i
// and dS_ij = P_ij (dP_ij - D_i), the gradients of L = sum(dout * out) are
//     dv_j = sum_i P_ij dout_i,   dk_j = scale sum_i dS_ij q_i,
//     dq_i = scale sum_j dS_ij k_j,
// summed over the query heads of each kv group for dk and dv
// (research.dws.rip/llm/kernels, section 01: outputs *and gradients* are
// what the kernels deliver; section 02: the backward decides the step).
//
// Three stream-ordered kernels, no atomics (bitwise reproducible):
//   1. preprocess (attn_aux.cu): D = rowsum(dout * out)
//   2. dK/dV pass: one CTA item = (segment, kv tile, kv head).  K and V stay
//      in shared memory; the CTA loops over the q tiles that can see the kv
//      tile and over the query heads of the group.  S^T = K Q^T and
//      dP^T = V dO^T land in TMEM; one thread per key row turns them into
//      P^T and dS^T (bf16, written back into the same TMEM columns), and
//      dV += P^T dO, dK += dS^T Q run with the A operand read from TMEM.
//   3. dQ pass: one CTA item = (segment, q tile, query head).  Q and dO stay
//      in shared memory; K/V tiles stream through a ring.  S = Q K^T and
//      dP = dO V^T in TMEM, dS (bf16) back into TMEM, dQ += dS K.
// Both passes visit only tiles the mask can see and use the same
// longest-first schedule as the forward.
#include <cuda_bf16.h>

#include "attn_internal.h"
#include "mask.cuh"
#include "ptx.cuh"
#include "sched.cuh"
#include "tiles.cuh"

namespace vsw {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Writes 32 fp32 accumulator columns of one row, scaled, as bf16 to global.
__device__ __forceinline__ void store_row32_bf16(void* dst_row, int c, const uint32_t (&r)[32], float mul) {
  uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dst_row) + c);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint4 pk;
    pk.x = pack_bf16x2(__uint_as_float(r[v * 8 + 0]) * mul, __uint_as_float(r[v * 8 + 1]) * mul);
    pk.y = pack_bf16x2(__uint_as_float(r[v * 8 + 2]) * mul, __uint_as_float(r[v * 8 + 3]) * mul);
    pk.z = pack_bf16x2(__uint_as_float(r[v * 8 + 4]) * mul, __uint_as_float(r[v * 8 + 5]) * mul);
    pk.w = pack_bf16x2(__uint_as_float(r[v * 8 + 6]) * mul, __uint_as_float(r[v * 8 + 7]) * mul);
    dst[v] = pk;
  }
}

// ============================================================== dK / dV pass
struct DkvCfg {
  static constexpr int kStages = 2;  // Q/dO tile pairs in flight
  static constexpr int kThreads = 256;
  static constexpr uint32_t kKOff = 0;
  static constexpr uint32_t kVOff = kTileBytes;
  static constexpr uint32_t kQOff = 2 * kTileBytes;  // stage s: Q at kQOff + 2s tiles, dO right after
  static constexpr uint32_t kSmemBytes = (2 + 2 * kStages) * kTileBytes + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
};

__global__ void __launch_bounds__(DkvCfg::kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                         const BwdParams p) {
  using C = DkvCfg;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ WorkItem items[kMaxItemsPerCta];
  __shared__ int item_counter, n_items;
  __shared__ __align__(8) uint64_t bar_kv_full, bar_kv_empty;
  __shared__ __align__(8) uint64_t bar_qdo_full[S], bar_qdo_empty[S];
  __shared__ __align__(8) uint64_t bar_s_full, bar_p_full, bar_mma_done, bar_acc_full;
  __shared__ __align__(8) uint64_t bar_stage[2];
  __shared__ __align__(16) float s_lse[2][128];
  __shared__ __align__(16) float s_delta[2][128];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t sK = sbase + C::kKOff, sV = sbase + C::kVOff, sQ0 = sbase + C::kQOff;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnParams& a = p.a;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_kv_full), 1);
    mbar_init(smem_u32(&bar_kv_empty), 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bar_qdo_full[s]), 1);
      mbar_init(smem_u32(&bar_qdo_empty[s]), 1);
    }
    mbar_init(smem_u32(&bar_s_full), 1);
    mbar_init(smem_u32(&bar_p_full), 128);
    mbar_init(smem_u32(&bar_mma_done), 1);
    mbar_init(smem_u32(&bar_acc_full), 1);
    mbar_init(smem_u32(&bar_stage[0]), 128);
    mbar_init(smem_u32(&bar_stage[1]), 128);
    fence_mbar_init();
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
    tma_prefetch_map(&tmDO);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 3) {
    int* cu = reinterpret_cast<int*>(gbase + C::kQOff);
    for (int s = lane; s <= a.nseg; s += 32) cu[s] = a.cu_seqlens[s];
    __syncwarp();
    const int n = build_schedule(cu, a.nseg, a.max_levels, a.hkv, true, items, kMaxItemsPerCta, &item_counter,
                                 blockIdx.x, gridDim.x);
    if (lane == 0) {
      n_items = n < 0 ? 0 : n;
      if (n < 0) atomicExch(a.status, 2);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int nit = n_items;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int cnt = 0;
      bool ok = true;
      for (int it = 0; it < nit && ok; ++it) {
        const WorkItem w = items[it];
        const int nb = num_tiles(w.seg_hi - w.seg_lo);
        const int k0 = w.seg_lo + w.blk * kTile;
        const int bl = last_q_tile(w.blk, nb, a.window);
        const int g = w.unit;
        if (it > 0 && !(ok = mbar_wait(smem_u32(&bar_kv_empty), (it - 1) & 1, &abort_flag, a.status))) break;
        mbar_arrive_expect_tx(smem_u32(&bar_kv_full), 2 * kTileBytes);
        tma_load_3d(sK, &tmK, smem_u32(&bar_kv_full), 0, g, k0);
        tma_load_3d(sK + kHalfTile, &tmK, smem_u32(&bar_kv_full), 64, g, k0);
        tma_load_3d(sV, &tmV, smem_u32(&bar_kv_full), 0, g, k0);
        tma_load_3d(sV + kHalfTile, &tmV, smem_u32(&bar_kv_full), 64, g, k0);
        for (int b = w.blk; b <= bl && ok; ++b) {
          const int q0 = w.seg_lo + b * kTile;
          for (int hh = 0; hh < a.group; ++hh) {
            const int h = g * a.group + hh;
            const int slot = cnt % S, use = cnt / S;
            if (use > 0 && !(ok = mbar_wait(smem_u32(&bar_qdo_empty[slot]), (use - 1) & 1, &abort_flag, a.status)))
              break;
            const uint32_t bar = smem_u32(&bar_qdo_full[slot]);
            const uint32_t sq = sQ0 + slot * 2 * kTileBytes, sdo = sq + kTileBytes;
            mbar_arrive_expect_tx(bar, 2 * kTileBytes);
            tma_load_3d(sq, &tmQ, bar, 0, h, q0);
            tma_load_3d(sq + kHalfTile, &tmQ, bar, 64, h, q0);
            tma_load_3d(sdo, &tmDO, bar, 0, h, q0);
            tma_load_3d(sdo + kHalfTile, &tmDO, bar, 64, h, q0);
            ++cnt;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_ss = make_idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idesc_ts = make_idesc_bf16(128, 128, 0, 1);
      int cnt = 0;
      bool ok = true;
      for (int it = 0; it < nit && ok; ++it) {
        const WorkItem w = items[it];
        const int nb = num_tiles(w.seg_hi - w.seg_lo);
        const int bl = last_q_tile(w.blk, nb, a.window);
        if (!(ok = mbar_wait(smem_u32(&bar_kv_full), it & 1, &abort_flag, a.status))) break;
        tc_fence_after();
        bool first = true;
        for (int b = w.blk; b <= bl && ok; ++b) {
          for (int hh = 0; hh < a.group; ++hh) {
            const int slot = cnt % S;
            if (!(ok = mbar_wait(smem_u32(&bar_qdo_full[slot]), (cnt / S) & 1, &abort_flag, a.status))) break;
            // The previous iteration's dV/dK MMAs read P^T/dS^T from the S/dP
            // columns; they must finish before S^T/dP^T are overwritten.
            if (cnt > 0 && !(ok = mbar_wait(smem_u32(&bar_mma_done), (cnt - 1) & 1, &abort_flag, a.status))) break;
            tc_fence_after();
            const uint32_t sq = sQ0 + slot * 2 * kTileBytes, sdo = sq + kTileBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + C::kColS, kmajor_desc(sK, kk), kmajor_desc(sq, kk), idesc_ss, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + C::kColDP, kmajor_desc(sV, kk), kmajor_desc(sdo, kk), idesc_ss, kk > 0);
            tc_commit(smem_u32(&bar_s_full));
            if (!(ok = mbar_wait(smem_u32(&bar_p_full), cnt & 1, &abort_flag, a.status))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + C::kColDV, tmem + C::kColS + kk * 8, mnmajor_desc(sdo, kk), idesc_ts,
                     (!first || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + C::kColDK, tmem + C::kColDP + kk * 8, mnmajor_desc(sq, kk), idesc_ts,
                     (!first || kk > 0) ? 1u : 0u);
            tc_commit(smem_u32(&bar_qdo_empty[slot]));
            tc_commit(smem_u32(&bar_mma_done));
            first = false;
            ++cnt;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&bar_acc_full));
        tc_commit(smem_u32(&bar_kv_empty));
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ elementwise
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key row of the kv tile
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    uint32_t s_cnt = 0;
    bool ok = true;
    for (int it = 0; it < nit && ok; ++it) {
      const WorkItem w = items[it];
      const int nb = num_tiles(w.seg_hi - w.seg_lo);
      const int k0 = w.seg_lo + w.blk * kTile;
      const int bl = last_q_tile(w.blk, nb, a.window);
      const int g = w.unit;
      const int j = k0 + row;  // this thread's key token
      for (int b = w.blk; b <= bl && ok; ++b) {
        const int q0 = w.seg_lo + b * kTile;
        for (int hh = 0; hh < a.group; ++hh) {
          const int h = g * a.group + hh;
          // Stage lse (log2 domain) and D of the tile's 128 queries.
          const int buf = s_cnt & 1;
          {
            const int iq = q0 + row;
            const bool in = token_in_range(iq, a.total);
            s_lse[buf][row] = in ? p.lse[(size_t)h * a.total + iq] * kLog2e : 0.f;
            s_delta[buf][row] = in ? p.delta[(size_t)h * a.total + iq] : 0.f;
          }
          // All 128 values staged before anyone reads them (bounded wait).
          mbar_arrive(smem_u32(&bar_stage[buf]));
          if (!(ok = mbar_wait(smem_u32(&bar_stage[buf]), (s_cnt >> 1) & 1, &abort_flag, a.status))) break;
          if (!(ok = mbar_wait(smem_u32(&bar_s_full), s_cnt & 1, &abort_flag, a.status))) break;
          ++s_cnt;
          tc_fence_after();
          int c_lo = 0, c_hi = kTile - 1;
          if (!tile_fully_visible_kv(k0, q0, w.seg_hi, a.window)) col_visible_rows(j, q0, w.seg_hi, a.window, c_lo, c_hi);
          float pr[128];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_base + C::kColS + c * 32, r);
            tmem_wait_ld(r);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 l4 = *reinterpret_cast<const float4*>(&s_lse[buf][c * 32 + e]);
              const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int col = c * 32 + e + u;
                const float x = ex2_approx(fmaf(__uint_as_float(r[e + u]), a.scale_log2, -lv[u]));
                pr[col] = (col >= c_lo && col <= c_hi) ? x : 0.f;
              }
            }
          }
          // P^T (bf16) over the S^T columns: 64 packed columns.
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) pk[e] = pack_bf16x2(pr[c * 64 + 2 * e], pr[c * 64 + 2 * e + 1]);
            tmem_st32(lane_base + C::kColS + c * 32, pk);
          }
          // dS^T = P^T (dP^T - D), written packed over the dP^T columns chunk by chunk.
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_base + C::kColDP + c * 32, r);
            tmem_wait_ld(r);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const int col = c * 32 + e;
              const float d0 = pr[col] * (__uint_as_float(r[e]) - s_delta[buf][col]);
              const float d1 = pr[col + 1] * (__uint_as_float(r[e + 1]) - s_delta[buf][col + 1]);
              pk[e >> 1] = pack_bf16x2(d0, d1);
            }
            tmem_st16(lane_base + C::kColDP + c * 16, pk);
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(smem_u32(&bar_p_full));
        }
      }
      if (!ok) break;
      // ---- epilogue: dV, dK (x scale) of this kv tile
      if (!(ok = mbar_wait(smem_u32(&bar_acc_full), it & 1, &abort_flag, a.status))) break;
      tc_fence_after();
      const bool valid = j < w.seg_hi && token_in_range(j, a.total);
      void* dv_row = static_cast<__nv_bfloat16*>(p.dv) + ((size_t)j * a.hkv + g) * kHeadDim;
      void* dk_row = static_cast<__nv_bfloat16*>(p.dk) + ((size_t)j * a.hkv + g) * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(lane_base + C::kColDV + c * 32, r);
        tmem_wait_ld(r);
        if (valid) store_row32_bf16(dv_row, c * 32, r, 1.f);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(lane_base + C::kColDK + c * 32, r);
        tmem_wait_ld(r);
        if (valid) store_row32_bf16(dk_row, c * 32, r, a.scale);
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ============================================================== dQ pass
struct DqCfg {
  static constexpr int kStages = 4;  // K/V tile slots
  static constexpr int kThreads = 256;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kDOOff = kTileBytes;
  static constexpr uint32_t kKVOff = 2 * kTileBytes;
  static constexpr uint32_t kSmemBytes = (2 + kStages) * kTileBytes + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;
};

__global__ void __launch_bounds__(DqCfg::kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const BwdParams p) {
  using C = DqCfg;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ WorkItem items[kMaxItemsPerCta];
  __shared__ int item_counter, n_items;
  __shared__ __align__(8) uint64_t bar_q_full, bar_q_empty;
  __shared__ __align__(8) uint64_t bar_kv_full[S], bar_kv_empty[S];
  __shared__ __align__(8) uint64_t bar_s_full, bar_p_full, bar_mma_done, bar_acc_full;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t sQ = sbase + C::kQOff, sDO = sbase + C::kDOOff, sKV = sbase + C::kKVOff;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnParams& a = p.a;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q_full), 1);
    mbar_init(smem_u32(&bar_q_empty), 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bar_kv_full[s]), 1);
      mbar_init(smem_u32(&bar_kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&bar_s_full), 1);
    mbar_init(smem_u32(&bar_p_full), 128);
    mbar_init(smem_u32(&bar_mma_done), 1);
    mbar_init(smem_u32(&bar_acc_full), 1);
    fence_mbar_init();
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
    tma_prefetch_map(&tmDO);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 3) {
    int* cu = reinterpret_cast<int*>(gbase + C::kKVOff);
    for (int s = lane; s <= a.nseg; s += 32) cu[s] = a.cu_seqlens[s];
    __syncwarp();
    const int n = build_schedule(cu, a.nseg, a.max_levels, a.hq, false, items, kMaxItemsPerCta, &item_counter,
                                 blockIdx.x, gridDim.x);
    if (lane == 0) {
      n_items = n < 0 ? 0 : n;
      if (n < 0) atomicExch(a.status, 2);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int nit = n_items;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int kv_cnt = 0;
      bool ok = true;
      for (int it = 0; it < nit && ok; ++it) {
        const WorkItem w = items[it];
        const int q0 = w.seg_lo + w.blk * kTile;
        const int n0 = first_kv_tile(w.blk, a.window);
        const int h = w.unit, g = h / a.group;
        if (it > 0 && !(ok = mbar_wait(smem_u32(&bar_q_empty), (it - 1) & 1, &abort_flag, a.status))) break;
        mbar_arrive_expect_tx(smem_u32(&bar_q_full), 2 * kTileBytes);
        tma_load_3d(sQ, &tmQ, smem_u32(&bar_q_full), 0, h, q0);
        tma_load_3d(sQ + kHalfTile, &tmQ, smem_u32(&bar_q_full), 64, h, q0);
        tma_load_3d(sDO, &tmDO, smem_u32(&bar_q_full), 0, h, q0);
        tma_load_3d(sDO + kHalfTile, &tmDO, smem_u32(&bar_q_full), 64, h, q0);
        for (int n = n0; n <= w.blk && ok; ++n) {
          const int k0 = w.seg_lo + n * kTile;
          for (int kv = 0; kv < 2; ++kv) {
            const int slot = kv_cnt % S, use = kv_cnt / S;
            if (use > 0 && !(ok = mbar_wait(smem_u32(&bar_kv_empty[slot]), (use - 1) & 1, &abort_flag, a.status)))
              break;
            const uint32_t bar = smem_u32(&bar_kv_full[slot]);
            mbar_arrive_expect_tx(bar, kTileBytes);
            const CUtensorMap* m = kv ? &tmV : &tmK;
            tma_load_3d(sKV + slot * kTileBytes, m, bar, 0, g, k0);
            tma_load_3d(sKV + slot * kTileBytes + kHalfTile, m, bar, 64, g, k0);
            ++kv_cnt;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_ss = make_idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idesc_ts = make_idesc_bf16(128, 128, 0, 1);
      int kv_cnt = 0, cnt = 0;
      bool ok = true;
      for (int it = 0; it < nit && ok; ++it) {
        const WorkItem w = items[it];
        const int n0 = first_kv_tile(w.blk, a.window);
        if (!(ok = mbar_wait(smem_u32(&bar_q_full), it & 1, &abort_flag, a.status))) break;
        tc_fence_after();
        for (int n = n0; n <= w.blk && ok; ++n) {
          const int slotK = kv_cnt % S;
          if (!(ok = mbar_wait(smem_u32(&bar_kv_full[slotK]), (kv_cnt / S) & 1, &abort_flag, a.status))) break;
          ++kv_cnt;
          const int slotV = kv_cnt % S;
          if (!(ok = mbar_wait(smem_u32(&bar_kv_full[slotV]), (kv_cnt / S) & 1, &abort_flag, a.status))) break;
          ++kv_cnt;
          // dS of the previous step (read by its dQ MMA) lives in the S columns.
          if (cnt > 0 && !(ok = mbar_wait(smem_u32(&bar_mma_done), (cnt - 1) & 1, &abort_flag, a.status))) break;
          tc_fence_after();
          const uint32_t kt = sKV + slotK * kTileBytes, vt = sKV + slotV * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::kColS, kmajor_desc(sQ, kk), kmajor_desc(kt, kk), idesc_ss, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::kColDP, kmajor_desc(sDO, kk), kmajor_desc(vt, kk), idesc_ss, kk > 0);
          tc_commit(smem_u32(&bar_s_full));
          tc_commit(smem_u32(&bar_kv_empty[slotV]));
          if (!(ok = mbar_wait(smem_u32(&bar_p_full), cnt & 1, &abort_flag, a.status))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::kColDQ, tmem + C::kColS + kk * 8, mnmajor_desc(kt, kk), idesc_ts,
                   (n > n0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(&bar_kv_empty[slotK]));
          tc_commit(smem_u32(&bar_mma_done));
          ++cnt;
        }
        if (!ok) break;
        tc_commit(smem_u32(&bar_acc_full));
        tc_commit(smem_u32(&bar_q_empty));
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ elementwise
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // query row of the q tile
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    uint32_t s_cnt = 0;
    bool ok = true;
    for (int it = 0; it < nit && ok; ++it) {
      const WorkItem w = items[it];
      const int q0 = w.seg_lo + w.blk * kTile;
      const int n0 = first_kv_tile(w.blk, a.window);
      const int h = w.unit;
      const int i = q0 + row;  // this thread's query token
      const bool valid = i < w.seg_hi && token_in_range(i, a.total);
      const float lse2 = valid ? p.lse[(size_t)h * a.total + i] * kLog2e : 0.f;
      const float dlt = valid ? p.delta[(size_t)h * a.total + i] : 0.f;
      for (int n = n0; n <= w.blk; ++n) {
        const int k0 = w.seg_lo + n * kTile;
        if (!(ok = mbar_wait(smem_u32(&bar_s_full), s_cnt & 1, &abort_flag, a.status))) break;
        ++s_cnt;
        tc_fence_after();
        int c_lo = 0, c_hi = kTile - 1;
        if (!tile_fully_visible(q0, k0, a.window)) row_visible_cols(i, k0, a.window, c_lo, c_hi);
        float pr[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(lane_base + C::kColS + c * 32, r);
          tmem_wait_ld(r);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = c * 32 + e;
            const float x = ex2_approx(fmaf(__uint_as_float(r[e]), a.scale_log2, -lse2));
            pr[col] = (col >= c_lo && col <= c_hi) ? x : 0.f;
          }
        }
        // dS = P (dP - D) -> bf16, packed over the S columns.
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(lane_base + C::kColDP + c * 32, r);
          tmem_wait_ld(r);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = c * 32 + e;
            pk[e >> 1] = pack_bf16x2(pr[col] * (__uint_as_float(r[e]) - dlt),
                                     pr[col + 1] * (__uint_as_float(r[e + 1]) - dlt));
          }
          tmem_st16(lane_base + C::kColS + c * 16, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_p_full));
      }
      if (!ok) break;
      if (!(ok = mbar_wait(smem_u32(&bar_acc_full), it & 1, &abort_flag, a.status))) break;
      tc_fence_after();
      void* dq_row = static_cast<__nv_bfloat16*>(p.dq) + ((size_t)i * a.hq + h) * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(lane_base + C::kColDQ + c * 32, r);
        tmem_wait_ld(r);
        if (valid) store_row32_bf16(dq_row, c * 32, r, a.scale);
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

long long persistent_grid(long long units, int num_sms) {
  long long grid = num_sms;
  const long long need = (units + kMaxItemsPerCta - 1) / kMaxItemsPerCta;
  if (need > grid) grid = need;
  if (units < grid) grid = units > 0 ? units : 1;
  return grid;
}

}  // namespace

int launch_bwd_dkdv(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmDO,
                    const BwdParams& p, int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)DkvCfg::kSmemBytes);
  if (e != cudaSuccess) return (int)e;
  const long long g = persistent_grid(upper_bound_tiles(p.a.total, p.a.nseg) * p.a.hkv, num_sms);
  attn_bwd_dkdv_kernel<<<(unsigned)g, DkvCfg::kThreads, DkvCfg::kSmemBytes, stream>>>(tmQ, tmK, tmV, tmDO, p);
  return (int)cudaGetLastError();
}

int launch_bwd_dq(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmDO,
                  const BwdParams& p, int num_sms, cudaStream_t stream) {
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DqCfg::kSmemBytes);
  if (e != cudaSuccess) return (int)e;
  const long long g = persistent_grid(upper_bound_tiles(p.a.total, p.a.nseg) * p.a.hq, num_sms);
  attn_bwd_dq_kernel<<<(unsigned)g, DqCfg::kThreads, DqCfg::kSmemBytes, stream>>>(tmQ, tmK, tmV, tmDO, p);
  return (int)cudaGetLastError();
}

}  // namespace vsw
