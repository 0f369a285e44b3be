// Forward pass of document-masked causal grouped-query attention on sm_103a.
//
// What it computes (research.dws.rip/llm/kernels, section 01 and Fig. 2):
// for each segment of the packed microbatch, each query head h and its
// key/value head g = h / (Hq/Hkv), softmax attention restricted to the keys
// that the mask in mask.cuh allows; it writes out (bf16) and the natural
// log-sum-exp of the scaled logits (fp32, [Hq, T]) for the backward pass.
//
// How (one persistent CTA per SM, warp-specialised):
//   warp 0        TMA producer: lane 1 streams the Q tiles of NQT heads per
//                 work unit through a ring of their own (the next unit's
//                 first head loads while the current unit runs), lane 0 the
//                 K_j, V_j tiles through a ring of slots
//   warp 1        MMA issuer: S_t = Q_t K_j^T (both operands in shared memory)
//                 and O_t += P_t V_j (P_t read from TMEM), fp32 accumulators
//                 in Tensor Memory
//   warp 2        owns the TMEM allocation
//   all threads   plan the CTA's longest-first work list in the prologue
//                 (plan.cuh); warp 3 alone when it does not fit (sched.cuh)
//   warpgroup 1+t online softmax of q tile t: one thread per query row reads
//                 its S row from TMEM, masks only tiles that straddle the mask
//                 edge, writes P (bf16) back over the first half of its S
//                 columns, rescales O in TMEM when the running max moves, and
//                 finally normalises O and stores out and lse.
// The NQT q tiles of a CTA are heads of the same group, so each K/V tile
// loaded from HBM/L2 feeds NQT heads.  Tiles that the mask hides completely
// are never loaded (the kv tile range comes from mask.cuh).
//
// P_t aliases S_t in TMEM.  This is safe because the MMA warp issues PV_t(j)
// (which reads P_t) before S_t(j+1) (which overwrites it) and tcgen05 MMAs of
// one thread execute in order; and the softmax only writes P_t(j) after it
// has read all of S_t(j).  When the softmax sees S_t(j+1) complete, PV_t(j)
// is complete too (the commit covers every earlier MMA), so O_t may then be
// rescaled without another barrier.
#include <cuda_bf16.h>

#include "attn_internal.h"
#include "mask.cuh"
#include "plan.cuh"
#include "ptx.cuh"
#include "sched.cuh"
#include "tiles.cuh"

namespace vsw {

namespace {

constexpr int kFwdMaxItems = 40;  // work units one CTA may own

template <int NQT>
struct FwdCfg {
  // Q tiles (one per head) go through a ring of their own: with NQT = 2 the
  // third slot takes the next item's first head while the current item runs,
  // and its second head follows as soon as the current first head's last S
  // MMA is done.  That leaves four K/V slots, so K(j+1) and V(j+1) can be in
  // flight while K(j)/V(j) are in use.
  static constexpr int kQSlots = NQT == 2 ? 3 : 2;
  static constexpr int kStages = NQT == 2 ? 4 : 5;     // K/V tile slots
  static constexpr int kThreads = 128 * (1 + NQT);
  static constexpr uint32_t kQOff = 0;                  // Q slot s at s tiles
  static constexpr uint32_t kKVOff = kQSlots * kTileBytes;
  static constexpr uint32_t kSmemBytes = kKVOff + kStages * kTileBytes + 1024;
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
  __shared__ WorkItem items[kFwdMaxItems];
  __shared__ int n_items;
  __shared__ __align__(8) uint64_t bar_q_full[C::kQSlots], bar_q_empty[C::kQSlots];
  __shared__ __align__(8) uint64_t bar_kv_full[S], bar_kv_empty[S];
  __shared__ __align__(8) uint64_t bar_s_full[NQT], bar_p_full[NQT], bar_o_done[NQT];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t sQ = sbase + C::kQOff, sKV = sbase + C::kKVOff;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnParams& a = p.a;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < C::kQSlots; ++s) {
      mbar_init(smem_u32(&bar_q_full[s]), 1);
      mbar_init(smem_u32(&bar_q_empty[s]), 1);
    }
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
  grid_dependency_wait();  // inputs written by earlier kernels are read after this
  // Work list: every thread plans (plan.cuh) in the not yet used tile region;
  // inputs too large for that fall back to the single-warp builder.
  const int planned = plan_schedule<false>(a.cu_seqlens, a.nseg, a.window, a.max_levels, a.hq / NQT, 0, items,
                                           kFwdMaxItems, reinterpret_cast<int*>(gbase),
                                           (int)((C::kSmemBytes - 1024) / 4), blockIdx.x, gridDim.x);
  if (planned == kPlanDoesNotFit) {
    if (warp == 3) {
      int* cu = reinterpret_cast<int*>(gbase + C::kKVOff);
      for (int s = lane; s <= a.nseg; s += 32) cu[s] = a.cu_seqlens[s];
      __syncwarp();
      const int n = build_schedule<false>(cu, a.nseg, a.window, a.max_levels, a.hq / NQT, 0, items, kFwdMaxItems,
                                          cu + kMaxSegments + 1, blockIdx.x, gridDim.x);
      if (lane == 0) {
        n_items = n < 0 ? 0 : n;
        if (n < 0) atomicExch(a.status, kStatusListOverflow);
      }
    }
  } else if (threadIdx.x == 0) {
    n_items = planned < 0 ? 0 : planned;
    if (planned < 0) atomicExch(a.status, kStatusListOverflow);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int nit = n_items;
  // With two softmax warpgroups, they take the registers the single-thread
  // roles do not need (launch: 168 x 384 threads; after: 104 x 128 +
  // 200 x 256, the same total, with no spills at these limits).
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (NQT == 2) regs_decrease<104>();
    // Lane 1 streams the Q tiles and lane 0 the K/V tiles, each through its
    // own ring: the next unit's Q tiles load as soon as their slots free up,
    // not after the last K/V load of the current unit.
    if (lane == 1) {
      int q_cnt = 0;
      bool ok = true;
      for (int it = 0; it < nit && ok; ++it) {
        const WorkItem w = items[it];
        const int q_lo = w.seg_lo + w.blk * kTile;
        for (int t = 0; t < NQT && ok; ++t, ++q_cnt) {
          const int slot = q_cnt % C::kQSlots, use = q_cnt / C::kQSlots;
          if (use > 0 && !(ok = mbar_wait(smem_u32(&bar_q_empty[slot]), (use - 1) & 1, &abort_flag, a.status)))
            break;
          const uint32_t qbar = smem_u32(&bar_q_full[slot]);
          mbar_arrive_expect_tx(qbar, kTileBytes);
          const int h = w.unit * NQT + t;
          const uint32_t dst = sQ + slot * kTileBytes;
          tma_load_3d(dst, &tmQ, qbar, 0, h, q_lo);
          tma_load_3d(dst + kHalfTile, &tmQ, qbar, 64, h, q_lo);
        }
      }
    } else if (lane == 0) {
      int kv_cnt = 0;
      bool ok = true;
      for (int it = 0; it < nit && ok; ++it) {
        const WorkItem w = items[it];
        const int n0 = w.t0;
        const int nt = w.t1 - w.t0 + 1;
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
    if (NQT == 2) regs_decrease<104>();
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idesc_pv = make_idesc_bf16(128, 128, 0, 1);
      int kv_cnt = 0, q_cnt = 0;
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
      // S_t = Q_t K^T into S_t; the Q slot of head t is released after its last S.
      auto issue_qk = [&](int t, int qs, int slotK, bool last) {
        const uint32_t d = tmem + t * 128;
        const uint32_t qt = sQ + qs * kTileBytes, kt = sKV + slotK * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(d, kmajor_desc(qt, kk), kmajor_desc(kt, kk), idesc_qk, kk > 0);
        tc_commit(smem_u32(&bar_s_full[t]));
        if (last) tc_commit(smem_u32(&bar_q_empty[qs]));
      };
      auto wait_q = [&](int& qs) -> bool {  // the next head's Q tile, in load order
        qs = q_cnt % C::kQSlots;
        const bool r = mbar_wait(smem_u32(&bar_q_full[qs]), (q_cnt / C::kQSlots) & 1, &abort_flag, a.status);
        ++q_cnt;
        tc_fence_after();
        return r;
      };
      // Units follow each other without a gap: S_t of the next unit's first kv
      // tile is issued right after PV_t of this unit's last one (it overwrites
      // P_t, which that PV read: in-order execution), so the softmax finds it
      // ready when it has finished this unit's epilogue.
      int qslot[NQT];
      if (nit > 0) {
        int slotK;
        for (int t = 0; t < NQT && ok; ++t) ok = wait_q(qslot[t]);
        if (ok) ok = wait_kv(slotK);
        if (ok) {
          const int nt0 = items[0].t1 - items[0].t0 + 1;
          for (int t = 0; t < NQT; ++t) issue_qk(t, qslot[t], slotK, nt0 == 1);
          tc_commit(smem_u32(&bar_kv_empty[slotK]));
        }
      }
      for (int it = 0; it < nit && ok; ++it) {
        const WorkItem w = items[it];
        const int nt = w.t1 - w.t0 + 1;
        const bool has_next = it + 1 < nit;
        const int nt_next = has_next ? items[it + 1].t1 - items[it + 1].t0 + 1 : 0;
        int qnext[NQT];
        for (int j = 0; j < nt && ok; ++j) {
          int slotV, slotK2 = -1;
          if (!(ok = wait_kv(slotV))) break;
          for (int t = 0; t < NQT && ok; ++t) {
            if (!(ok = mbar_wait(smem_u32(&bar_p_full[t]), p_cnt[t] & 1, &abort_flag, a.status))) break;
            ++p_cnt[t];
            tc_fence_after();
            const uint32_t d = tmem + C::kOCol + t * 128;
            const uint32_t vt = sKV + slotV * kTileBytes;
            // O_t += P_t V: P_t (bf16, 64 packed columns over S_t) is the A operand.
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(d, tmem + t * 128 + kk * 8, mnmajor_desc(vt, kk), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
            if (j + 1 == nt) tc_commit(smem_u32(&bar_o_done[t]));
            // V(j) is free once the last head's PV has read it.
            if (t == NQT - 1) tc_commit(smem_u32(&bar_kv_empty[slotV]));
            if (j + 1 < nt) {
              if (t == 0 && !(ok = wait_kv(slotK2))) break;
              issue_qk(t, qslot[t], slotK2, j + 2 == nt);
            } else if (has_next) {
              if (t == 0 && !(ok = wait_kv(slotK2))) break;
              if (!(ok = wait_q(qnext[t]))) break;
              issue_qk(t, qnext[t], slotK2, nt_next == 1);
            }
          }
          if (!ok) break;
          if (slotK2 >= 0) tc_commit(smem_u32(&bar_kv_empty[slotK2]));
        }
        if (has_next)
          for (int t = 0; t < NQT; ++t) qslot[t] = qnext[t];
      }
    }
  } else if (warp < 4) {
    if (NQT == 2) regs_decrease<104>();
    if (warp == 3 && blockIdx.x == 0) report_long_segments(a);
  } else {
    // ------------------------------------------------------------ softmax
    if (NQT == 2) regs_increase<200>();
    const int t = (warp >> 2) - 1;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    const uint32_t tS = lane_base + t * 128;
    const uint32_t tO = lane_base + C::kOCol + t * 128;
    const uint64_t scale2 = f2_pack(a.scale_log2, a.scale_log2);
    uint32_t s_cnt = 0;
    bool ok = true;
    for (int it = 0; it < nit && ok; ++it) {
      const WorkItem w = items[it];
      const int q_lo = w.seg_lo + w.blk * kTile;
      const int n0 = w.t0;
      const int nt = w.t1 - w.t0 + 1;
      const int h = w.unit * NQT + t;
      const int i = q_lo + row;  // this thread's query token
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        const int k0 = w.seg_lo + (n0 + j) * kTile;
        if (!(ok = mbar_wait_warp(smem_u32(&bar_s_full[t]), s_cnt & 1, &abort_flag, a.status))) break;
        ++s_cnt;
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld128_wait(tS, sr);
        float* s = reinterpret_cast<float*>(sr);
        if (!tile_fully_visible(q_lo, k0, a.window)) {
          int lo_rel, hi_rel;
          row_visible_cols(i, k0, a.window, lo_rel, hi_rel);
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c < lo_rel || c > hi_rel) s[c] = -INFINITY;
        }
        // Row max: a tree of three-input maxima.
        float mx[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) mx[e] = fmax3(s[8 * e], s[8 * e + 1], s[8 * e + 2]);
#pragma unroll
        for (int e = 0; e < 16; ++e) mx[e] = fmax3(mx[e], s[8 * e + 3], s[8 * e + 4]);
#pragma unroll
        for (int e = 0; e < 16; ++e) mx[e] = fmax3(mx[e], s[8 * e + 5], s[8 * e + 6]);
#pragma unroll
        for (int e = 0; e < 16; ++e) mx[e] = fmaxf(mx[e], s[8 * e + 7]);
#pragma unroll
        for (int e = 0; e < 5; ++e) mx[e] = fmax3(mx[e], mx[e + 5], mx[e + 10]);
        const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[15]), -INFINITY) * a.scale_log2;
        // Lazy rescaling: the reference max moves only when the tile max
        // exceeds it by more than 8 (log2 units), so P stays <= 2^8 and O is
        // rescaled in TMEM only on those (rare) tiles.  out = O / l and lse
        // use the same reference, so the result is exact.
        const bool bump = mt > m + 8.f;
        const float m_new = bump ? mt : m;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = bump ? ex2_approx(m - m_use) : 1.f;
        const uint64_t negm2 = f2_pack(-m_use, -m_use);
        uint64_t rs2[4] = {0, 0, 0, 0};
        // p = exp2(s * scale*log2e - m), packed to bf16 pairs 32 at a time and
        // stored over the first 64 columns of S_t.
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = 64 * h2 + 2 * e;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), scale2, negm2), x0, x1);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            rs2[e & 3] = f2_add(rs2[e & 3], f2_pack(p0, p1));
            pk[e] = pack_bf16x2(p0, p1);
          }
          tmem_st32(tS + 32 * h2, pk);
        }
        float r0, r1, r2, r3, r4, r5, r6, r7;
        f2_unpack(rs2[0], r0, r1);
        f2_unpack(rs2[1], r2, r3);
        f2_unpack(rs2[2], r4, r5);
        f2_unpack(rs2[3], r6, r7);
        const float rs = ((r0 + r1) + (r2 + r3)) + ((r4 + r5) + (r6 + r7));
        l = l * alpha + rs;
        m = m_new;
        // PV of the previous tile is complete here: the S commit just waited on
        // was issued after it.  Rescale O only where the reference moved.
        if (j > 0 && __any_sync(0xffffffffu, bump)) {
          const uint64_t alpha2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tmem_ld32(tO + c * 32, r);
            tmem_wait_ld(r);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float y0, y1;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), alpha2), y0, y1);
              r[e] = __float_as_uint(y0);
              r[e + 1] = __float_as_uint(y1);
            }
            tmem_st32(tO + c * 32, r);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_p_full[t]));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> out (bf16), lse
      if (!(ok = mbar_wait_warp(smem_u32(&bar_o_done[t]), it & 1, &abort_flag, a.status))) break;
      tc_fence_after();
      const bool valid = i < w.seg_hi && token_in_range(i, a.total);
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      void* out_row = static_cast<__nv_bfloat16*>(p.out) + i * p.out_st.token + h * p.out_st.head;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + c * 32, r);
        tmem_wait_ld(r);
        store_rows32_bf16(out_row, p.out_st.token * 2, c * 32, r, inv_l, valid);
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
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<NQT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)C::kSmemBytes);
  if (e != cudaSuccess) return (int)e;
  const long long units = upper_bound_tiles(p.a.total, p.a.nseg) * (p.a.hq / NQT);
  long long grid = num_sms;
  const long long need = (units + kFwdMaxItems - 1) / kFwdMaxItems;
  if (need > grid) grid = need;
  if (units < grid) grid = units > 0 ? units : 1;
  return (int)launch_pdl(attn_fwd_kernel<NQT>, dim3((unsigned)grid), dim3(C::kThreads), C::kSmemBytes, stream, tmQ,
                         tmK, tmV, p);
}

}  // namespace

int launch_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const FwdParams& p,
               int num_sms, cudaStream_t stream) {
  if ((p.a.group % 2) == 0) return launch_fwd_t<2>(tmQ, tmK, tmV, p, num_sms, stream);
  return launch_fwd_t<1>(tmQ, tmK, tmV, p, num_sms, stream);
}

}  // namespace vsw
