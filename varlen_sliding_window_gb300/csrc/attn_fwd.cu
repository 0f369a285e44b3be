// Forward pass of document-masked causal grouped-query attention on sm_103a.
//
// What it computes (research.dws.rip/llm/kernels, section 01 and Fig. 2):
// for each segment of the packed microbatch, each query head h and its
// key/value head g = h / (Hq/Hkv), softmax attention restricted to the keys
// that the mask in mask.cuh allows; it writes out (bf16) and the natural
// log-sum-exp of the scaled logits (fp32, [Hq, T]) for the backward pass.
//
// How (one persistent CTA per SM, warp-specialised):
//   warp 0        TMA producer: Q tiles of NQT heads, then K_j, V_j tiles
//                 through a ring of shared-memory slots
//   warp 1        MMA issuer: S_t = Q_t K_j^T and O_t += P_t V_j with tcgen05,
//                 accumulators in Tensor Memory
//   warp 2        owns the TMEM allocation
//   warp 3        builds the CTA's longest-first work list (sched.cuh)
//   warpgroup 1+t online softmax of q tile t: one thread per query row reads
//                 its S row from TMEM, masks only tiles that straddle the mask
//                 edge, rescales O in TMEM when the running max moves, writes
//                 P (bf16) to shared memory for the PV MMA, and finally
//                 normalises O and stores out and lse.
// The NQT q tiles of a CTA are heads of the same group, so each K/V tile
// loaded from HBM/L2 feeds NQT heads.  Tiles that the mask hides completely
// are never loaded (the kv tile range comes from mask.cuh).
#include <cuda_bf16.h>

#include "attn_internal.h"
#include "mask.cuh"
#include "ptx.cuh"
#include "sched.cuh"
#include "tiles.cuh"

namespace vsw {

namespace {

template <int NQT>
struct FwdCfg {
  static constexpr int kStages = NQT == 2 ? 3 : 4;
  static constexpr int kThreads = 128 * (1 + NQT);
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKVOff = NQT * kTileBytes;
  static constexpr uint32_t kPOff = kKVOff + kStages * kTileBytes;
  static constexpr uint32_t kSmemBytes = kPOff + NQT * kTileBytes + 1024;
  static constexpr uint32_t kTmemCols = NQT == 2 ? 512 : 256;
  static constexpr uint32_t kOCol = NQT * 128;  // O accumulators follow the S tiles
};

template <int NQT>
__global__ void __launch_bounds__(FwdCfg<NQT>::kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<NQT>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ WorkItem items[kMaxItemsPerCta];
  __shared__ int item_counter;
  __shared__ int n_items;
  __shared__ __align__(8) uint64_t bar_q_full, bar_q_empty;
  __shared__ __align__(8) uint64_t bar_kv_full[S], bar_kv_empty[S];
  __shared__ __align__(8) uint64_t bar_s_full[NQT], bar_p_full[NQT], bar_o_done[NQT];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t sQ = sbase + C::kQOff, sKV = sbase + C::kKVOff, sP = sbase + C::kPOff;
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
    for (int t = 0; t < NQT; ++t) {
      mbar_init(smem_u32(&bar_s_full[t]), 1);
      mbar_init(smem_u32(&bar_p_full[t]), 128);
      mbar_init(smem_u32(&bar_o_done[t]), 1);
    }
    fence_mbar_init();
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 3) {
    // cu_seqlens is staged in the (not yet used) P region.
    int* cu = reinterpret_cast<int*>(gbase + C::kPOff);
    for (int s = lane; s <= a.nseg; s += 32) cu[s] = a.cu_seqlens[s];
    __syncwarp();
    const int n = build_schedule(cu, a.nseg, a.max_levels, a.hq / NQT, false, items, kMaxItemsPerCta,
                                 &item_counter, blockIdx.x, gridDim.x);
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
        const int q_lo = w.seg_lo + w.blk * kTile;
        const int n0 = first_kv_tile(w.blk, a.window);
        const int nt = w.blk - n0 + 1;
        if (it > 0 && !(ok = mbar_wait(smem_u32(&bar_q_empty), (it - 1) & 1, &abort_flag, a.status))) break;
        mbar_arrive_expect_tx(smem_u32(&bar_q_full), NQT * kTileBytes);
        for (int t = 0; t < NQT; ++t) {
          const int h = w.unit * NQT + t;
          tma_load_3d(sQ + t * kTileBytes, &tmQ, smem_u32(&bar_q_full), 0, h, q_lo);
          tma_load_3d(sQ + t * kTileBytes + kHalfTile, &tmQ, smem_u32(&bar_q_full), 64, h, q_lo);
        }
        const int g = (w.unit * NQT) / a.group;
        for (int j = 0; j < nt && ok; ++j) {
          const int k0 = w.seg_lo + (n0 + j) * kTile;
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
      constexpr uint32_t idesc_qk = make_idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idesc_pv = make_idesc_bf16(128, 128, 0, 1);
      int kv_cnt = 0;
      uint32_t p_cnt[NQT];
      for (int t = 0; t < NQT; ++t) p_cnt[t] = 0;
      bool ok = true;
      auto wait_kv = [&](int& slot) -> bool {
        slot = kv_cnt % S;
        const bool r = mbar_wait(smem_u32(&bar_kv_full[slot]), (kv_cnt / S) & 1, &abort_flag, a.status);
        ++kv_cnt;
        tc_fence_after();
        return r;
      };
      auto issue_qk = [&](int t, int slotK) {
        const uint32_t d = tmem + t * 128;
        const uint32_t qt = sQ + t * kTileBytes, kt = sKV + slotK * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(d, kmajor_desc(qt, kk), kmajor_desc(kt, kk), idesc_qk, kk > 0);
        tc_commit(smem_u32(&bar_s_full[t]));
      };
      for (int it = 0; it < nit && ok; ++it) {
        const WorkItem w = items[it];
        const int n0 = first_kv_tile(w.blk, a.window);
        const int nt = w.blk - n0 + 1;
        if (!(ok = mbar_wait(smem_u32(&bar_q_full), it & 1, &abort_flag, a.status))) break;
        tc_fence_after();
        int slotK;
        if (!(ok = wait_kv(slotK))) break;
        for (int t = 0; t < NQT; ++t) issue_qk(t, slotK);
        tc_commit(smem_u32(&bar_kv_empty[slotK]));
        for (int j = 0; j < nt && ok; ++j) {
          int slotV, slotK2 = -1;
          if (!(ok = wait_kv(slotV))) break;
          for (int t = 0; t < NQT && ok; ++t) {
            if (!(ok = mbar_wait(smem_u32(&bar_p_full[t]), p_cnt[t] & 1, &abort_flag, a.status))) break;
            ++p_cnt[t];
            tc_fence_after();
            const uint32_t d = tmem + C::kOCol + t * 128;
            const uint32_t pt = sP + t * kTileBytes, vt = sKV + slotV * kTileBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(d, kmajor_desc(pt, kk), mnmajor_desc(vt, kk), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
            tc_commit(smem_u32(&bar_o_done[t]));
            if (j + 1 < nt) {
              if (t == 0 && !(ok = wait_kv(slotK2))) break;
              issue_qk(t, slotK2);
            }
          }
          if (!ok) break;
          tc_commit(smem_u32(&bar_kv_empty[slotV]));
          if (j + 1 < nt) tc_commit(smem_u32(&bar_kv_empty[slotK2]));
        }
        if (ok) tc_commit(smem_u32(&bar_q_empty));
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int t = (warp >> 2) - 1;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    const uint32_t tS = lane_base + t * 128;
    const uint32_t tO = lane_base + C::kOCol + t * 128;
    const uint32_t pT = sP + t * kTileBytes;
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ok = true;
    for (int it = 0; it < nit && ok; ++it) {
      const WorkItem w = items[it];
      const int q_lo = w.seg_lo + w.blk * kTile;
      const int n0 = first_kv_tile(w.blk, a.window);
      const int nt = w.blk - n0 + 1;
      const int h = w.unit * NQT + t;
      const int i = q_lo + row;  // this thread's query token
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        const int k0 = w.seg_lo + (n0 + j) * kTile;
        if (!(ok = mbar_wait(smem_u32(&bar_s_full[t]), s_cnt & 1, &abort_flag, a.status))) break;
        ++s_cnt;
        tc_fence_after();
        float s[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tS + c * 32, r);
          tmem_wait_ld(r);
#pragma unroll
          for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(r[e]);
        }
        if (!tile_fully_visible(q_lo, k0, a.window)) {
          int lo_rel, hi_rel;
          row_visible_cols(i, k0, a.window, lo_rel, hi_rel);
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c < lo_rel || c > hi_rel) s[c] = -INFINITY;
        }
        float mx = s[0];
#pragma unroll
        for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
        const float m_new = fmaxf(m, mx * a.scale_log2);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2_approx(m - m_use);
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          s[c] = ex2_approx(fmaf(s[c], a.scale_log2, -m_use));
          rs += s[c];
        }
        if (j > 0) {
          // PV of the previous tile must be done before O is rescaled and P overwritten.
          if (!(ok = mbar_wait(smem_u32(&bar_o_done[t]), o_cnt & 1, &abort_flag, a.status))) break;
          ++o_cnt;
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t r[32];
              tmem_ld32(tO + c * 32, r);
              tmem_wait_ld(r);
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              tmem_st32(tO + c * 32, r);
            }
            tmem_wait_st();
          }
        }
        l = l * alpha + rs;
        m = m_new;
        // P (bf16) into the 128-byte-swizzled K-major layout the MMA reads.
#pragma unroll
        for (int c8 = 0; c8 < 16; ++c8)
          st_shared_v4(swizzled_chunk(pT, row, c8), pack_bf16x2(s[c8 * 8 + 0], s[c8 * 8 + 1]),
                       pack_bf16x2(s[c8 * 8 + 2], s[c8 * 8 + 3]), pack_bf16x2(s[c8 * 8 + 4], s[c8 * 8 + 5]),
                       pack_bf16x2(s[c8 * 8 + 6], s[c8 * 8 + 7]));
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_p_full[t]));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> out (bf16), lse
      if (!(ok = mbar_wait(smem_u32(&bar_o_done[t]), o_cnt & 1, &abort_flag, a.status))) break;
      ++o_cnt;
      tc_fence_after();
      const bool valid = i < w.seg_hi && token_in_range(i, a.total);
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                            ((size_t)i * a.hq + h) * kHeadDim);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + c * 32, r);
        tmem_wait_ld(r);
        if (valid) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(r[v * 8 + 0]) * inv_l, __uint_as_float(r[v * 8 + 1]) * inv_l);
            pk.y = pack_bf16x2(__uint_as_float(r[v * 8 + 2]) * inv_l, __uint_as_float(r[v * 8 + 3]) * inv_l);
            pk.z = pack_bf16x2(__uint_as_float(r[v * 8 + 4]) * inv_l, __uint_as_float(r[v * 8 + 5]) * inv_l);
            pk.w = pack_bf16x2(__uint_as_float(r[v * 8 + 6]) * inv_l, __uint_as_float(r[v * 8 + 7]) * inv_l);
            dst[c * 4 + v] = pk;
          }
        }
      }
      if (valid) p.lse[(size_t)h * a.total + i] = (m + __log2f(l)) * 0.69314718055994531f;
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

template <int NQT>
int launch_fwd_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const FwdParams& p,
                 int num_sms, cudaStream_t stream) {
  using C = FwdCfg<NQT>;
  static bool attr_set = false;  // per process; the attribute is per function
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<NQT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::kSmemBytes);
    if (e != cudaSuccess) return (int)e;
    attr_set = true;
  }
  const long long units = upper_bound_tiles(p.a.total, p.a.nseg) * (p.a.hq / NQT);
  long long grid = num_sms;
  const long long need = (units + kMaxItemsPerCta - 1) / kMaxItemsPerCta;
  if (need > grid) grid = need;
  if (units < grid) grid = units > 0 ? units : 1;
  attn_fwd_kernel<NQT><<<(unsigned)grid, C::kThreads, C::kSmemBytes, stream>>>(tmQ, tmK, tmV, p);
  return (int)cudaGetLastError();
}

}  // namespace

int launch_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const FwdParams& p,
               int num_sms, cudaStream_t stream) {
  if ((p.a.group % 2) == 0) return launch_fwd_t<2>(tmQ, tmK, tmV, p, num_sms, stream);
  return launch_fwd_t<1>(tmQ, tmK, tmV, p, num_sms, stream);
}

}  // namespace vsw
