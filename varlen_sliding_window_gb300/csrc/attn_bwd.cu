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
//      tile and over the query heads of the group.
//   3. dQ pass: one CTA item = (segment, q tile, query head).  Q and dO stay
//      in shared memory; K/V tiles stream through a ring.
//
// TMEM holds the fp32 accumulators of the MMAs (128 lanes x 512 columns):
//   dK/dV pass: S^T, dP^T (N = 128 queries), dV, dK.  The two elementwise
//     warpgroups split each tile's 128 query columns.  S^T and dP^T complete
//     separately: P^T (the exp2 work) is computed while dP^T still runs, and
//     both bf16 P^T and dS^T go back over the dP^T columns, so S^T of the
//     next pair runs as soon as S^T has been read into registers.  dV and dK
//     of a 64-query half start as soon as that half is back in TMEM.
//   dQ pass: two S buffers, dP, dQ.  S of the next kv tile is computed while
//     the elementwise warpgroups work on the current one, and dP is released
//     as soon as it has been read into registers.
// bf16 operands (P^T, dS^T, dS) go back over fp32 columns the same warps have
// already read and feed the next MMA as its A operand straight from TMEM.
// tcgen05 MMAs issued by one thread execute in order, so an MMA that
// overwrites such columns always runs after the MMAs that read them.  Measured on GB300: a 128x64x16 MMA takes as long as a 128x128x16 one,
// so every S/dP MMA here uses N = 128.
#include <cuda_bf16.h>

#include "attn_internal.h"
#include "claim.cuh"
#include "mask.cuh"
#include "plan.cuh"
#include "ptx.cuh"
#include "sched.cuh"
#include "tiles.cuh"

namespace vsw {

static_assert(sizeof(WorkItem) == kWorkItemBytes, "the workspace sizes its unit lists with this");

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// One TMEM load of 64 consecutive columns (two x32 loads, one wait).
__device__ __forceinline__ void tmem_ld64_wait(uint32_t taddr, uint32_t (&r)[64]) {
  uint32_t(&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
  uint32_t(&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[32]);
  tmem_ld32(taddr, lo);
  tmem_ld32(taddr + 32, hi);
  tmem_wait_ld(lo);
  tmem_wait_ld(hi);
}

// Role split of the 384-thread backward CTAs: warpgroup 0 holds the producer,
// MMA, TMEM and scheduler warps (few registers), warpgroups 1 and 2 do the
// elementwise work (launch 168 x 384 = 104 x 128 + 200 x 256 registers).
constexpr int kBwdThreads = 384;
constexpr int kBwdMaxItems = 96;  // work units one CTA may own

// ============================================================== dK / dV pass
struct DkvCfg {
  static constexpr int kStages = 2;  // Q/dO tile pairs in flight
  static constexpr uint32_t kKOff = 0;
  static constexpr uint32_t kVOff = kTileBytes;
  static constexpr uint32_t kQOff = 2 * kTileBytes;  // stage s: Q at kQOff + 2s tiles, dO right after
  // Extra k-step of S^T and dP^T (tiles.cuh): a block of ones (the A side, for
  // K and V) and per stage the query-side blocks holding -lse/scale (with Q)
  // and -D (with dO), each split into a bf16 high and low part, so the MMAs
  // deliver s - lse/scale and dP - D directly.
  static constexpr uint32_t kAugOff = (2 + 2 * kStages) * kTileBytes;
  static constexpr uint32_t kOnesOff = kAugOff;
  static constexpr uint32_t kQxOff = kAugOff + kAugBytes;                 // + s * kAugBytes
  static constexpr uint32_t kDOxOff = kAugOff + (1 + kStages) * kAugBytes;  // + s * kAugBytes
  static constexpr uint32_t kAugEnd = kAugOff + (1 + 2 * kStages) * kAugBytes;
  static constexpr uint32_t kSmemBytes = kAugEnd + 1024;
  static constexpr uint32_t kTmemCols = 512;
  // S^T, dP^T (128 columns each, fp32; bf16 dS^T and P^T over dP^T), dV, dK.
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
};

__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                         const BwdParams p) {
  using C = DkvCfg;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ WorkItem items[kBwdMaxItems];
  __shared__ int n_items;
  // Items in flight, handed from the claiming warp to the other roles.
  __shared__ WorkItem ring[2];
  __shared__ __align__(8) uint64_t ring_full[2], ring_taken[2], ring_empty[2];
  __shared__ int claim_mode, n_units_s;
  __shared__ int* claim_words;
  __shared__ __align__(8) uint64_t bar_kv_full, bar_kv_empty;
  __shared__ __align__(8) uint64_t bar_qdo_full[S], bar_qdo_empty[S];
  // s_full[0]: S^T done, s_full[1]: dP^T done; s_free: both warpgroups have
  // read S^T into registers; ds_full[x]: warpgroup x has written its half of
  // P^T and dS^T.
  __shared__ __align__(8) uint64_t bar_s_full[2], bar_s_free, bar_ds_full[2];
  __shared__ __align__(8) uint64_t bar_acc_full, bar_acc_empty;
  __shared__ __align__(8) uint64_t bar_chain[2];
  __shared__ int chain_last[2];
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
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&bar_s_full[x]), 1);
      mbar_init(smem_u32(&bar_ds_full[x]), 128);
    }
    mbar_init(smem_u32(&bar_s_free), 256);
    mbar_init(smem_u32(&bar_acc_full), 1);
    mbar_init(smem_u32(&bar_acc_empty), 256);
    mbar_init(smem_u32(&bar_chain[0]), 128);
    mbar_init(smem_u32(&bar_chain[1]), 128);
    for (int r = 0; r < 2; ++r) {
      mbar_init(smem_u32(&ring_full[r]), 1);
      mbar_init(smem_u32(&ring_taken[r]), 1);
      mbar_init(smem_u32(&ring_empty[r]), 10);  // the producer warp, the MMA thread, the 8 elementwise warps
    }
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
  // Inputs written by earlier kernels (and the unit list of this backward's
  // planning kernel) are read after the wait.  With a fresh list every CTA
  // claims units at run time (claim.cuh); otherwise it plans its own share.
  grid_dependency_wait();
  if (threadIdx.x == 0) {
    int* cw = p.sched;
    claim_mode = cw ? claim_ready(cw) : 0;
    n_units_s = claim_mode ? __ldcg(cw + 3) : 0;
    claim_words = claim_mode ? cw : nullptr;
    n_items = 0;
  }
  __syncthreads();
  const int planned = claim_mode ? 0
                                 : plan_schedule<true>(a.cu_seqlens, a.nseg, a.window, a.max_levels, a.hkv,
                                                       p.chains_max, items, kBwdMaxItems, reinterpret_cast<int*>(gbase),
                                                       (int)(C::kAugOff / 4), blockIdx.x, gridDim.x);
  if (planned == kPlanDoesNotFit) {
    if (warp == 3) {
      int* cu = reinterpret_cast<int*>(gbase + C::kQOff);
      for (int s = lane; s <= a.nseg; s += 32) cu[s] = a.cu_seqlens[s];
      __syncwarp();
      const int n = build_schedule<true>(cu, a.nseg, a.window, a.max_levels, a.hkv, p.chains_max, items,
                                         kBwdMaxItems, cu + kMaxSegments + 1, blockIdx.x, gridDim.x);
      if (lane == 0) {
        n_items = n < 0 ? 0 : n;
        if (n < 0) atomicExch(a.status, kStatusListOverflow);
      }
    }
  } else if (threadIdx.x == 0 && !claim_mode) {
    n_items = planned < 0 ? 0 : planned;
    if (planned < 0) atomicExch(a.status, kStatusListOverflow);
  }
  // Extra k-step blocks (after the planner, whose scratch ends at kAugOff):
  // the ones block gets 1.0 in columns 0 and 1 of every row, the per-stage
  // blocks start at zero and only their columns 0 and 1 change later.
  if (threadIdx.x < 128) {
    const uint32_t ones = sbase + C::kOnesOff;
    const int r = threadIdx.x;
    const uint32_t c0 = aug_chunk0(ones, r);
    st_shared_v4(c0, 0x3F803F80u, 0u, 0u, 0u);
    st_shared_v4(c0 ^ 16u, 0u, 0u, 0u, 0u);
  }
  for (uint32_t off = C::kQxOff + 16u * threadIdx.x; off < C::kAugEnd; off += 16u * blockDim.x)
    st_shared_v4(sbase + off, 0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int nit = n_items;
  // The dQ kernel that follows in the same backward reads nothing this kernel
  // writes: let it take the SMs this grid frees (it waits for this grid to
  // finish only before it exits).
  grid_dependents_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // TMA for K, V (per item) and Q, dO (per q tile and head); the warp's 32
    // lanes write the stage's query-side extra k-step blocks (-lse/scale and
    // -D of its 128 queries, as bf16 high + low parts).
    regs_decrease<104>();
    const float inv_scale = 1.f / a.scale;
    int cnt = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int rs = it & 1;
      if (!(ok = mbar_wait_warp(smem_u32(&ring_full[rs]), (it >> 1) & 1, &abort_flag, a.status))) break;
      const WorkItem w = ring[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ring_empty[rs]));
      if (w.blk < 0) break;
      const int k0 = w.seg_lo + w.blk * kTile;
      const int g = w.unit;
      if (lane == 0) {
        if (it > 0) ok = mbar_wait(smem_u32(&bar_kv_empty), (it - 1) & 1, &abort_flag, a.status);
        if (ok) {
          mbar_arrive_expect_tx(smem_u32(&bar_kv_full), 2 * kTileBytes);
          tma_load_3d(sK, &tmK, smem_u32(&bar_kv_full), 0, g, k0);
          tma_load_3d(sK + kHalfTile, &tmK, smem_u32(&bar_kv_full), 64, g, k0);
          tma_load_3d(sV, &tmV, smem_u32(&bar_kv_full), 0, g, k0);
          tma_load_3d(sV + kHalfTile, &tmV, smem_u32(&bar_kv_full), 64, g, k0);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      for (int b = w.t0; b <= w.t1 && ok; ++b) {
        const int q0 = w.seg_lo + b * kTile;
        for (int hh = 0; hh < a.group && ok; ++hh) {
          const int h = g * a.group + hh;
          const int slot = cnt % S, use = cnt / S;
          // This stage's lse and D loads go out before the wait for its slot.
          float lv[4], dlv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int iq = q0 + lane + 32 * e;
            const bool in = token_in_range(iq, a.total);
            lv[e] = in ? __ldg(p.lse + (size_t)h * a.total + iq) : 0.f;
            dlv[e] = in ? __ldg(p.delta + (size_t)h * a.total + iq) : 0.f;
          }
          if (use > 0) {
            if (lane == 0) ok = mbar_wait(smem_u32(&bar_qdo_empty[slot]), (use - 1) & 1, &abort_flag, a.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = lane + 32 * e;
            const float L = -lv[e] * inv_scale, Dn = -dlv[e];
            const float L_hi = __bfloat162float(__float2bfloat16_rn(L));
            const float D_hi = __bfloat162float(__float2bfloat16_rn(Dn));
            st_shared_u32(aug_chunk0(sbase + C::kQxOff + slot * kAugBytes, c), pack_bf16x2(L_hi, L - L_hi));
            st_shared_u32(aug_chunk0(sbase + C::kDOxOff + slot * kAugBytes, c), pack_bf16x2(D_hi, Dn - D_hi));
          }
          fence_proxy_async_smem();  // the MMA reads these blocks through the async proxy
          __syncwarp();
          if (lane == 0) {
            const uint32_t bar = smem_u32(&bar_qdo_full[slot]);
            const uint32_t sq = sQ0 + slot * 2 * kTileBytes, sdo = sq + kTileBytes;
            mbar_arrive_expect_tx(bar, 2 * kTileBytes);
            tma_load_3d(sq, &tmQ, bar, 0, h, q0);
            tma_load_3d(sq + kHalfTile, &tmQ, bar, 64, h, q0);
            tma_load_3d(sdo, &tmDO, bar, 0, h, q0);
            tma_load_3d(sdo + kHalfTile, &tmDO, bar, 64, h, q0);
          }
          ++cnt;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    regs_decrease<104>();
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, 0, 0);   // S^T, dP^T: 128 keys x 128 queries
      constexpr uint32_t idesc_g = make_idesc_bf16(128, 128, 0, 1);   // dV, dK: 128 keys x 128 dims
      const uint32_t sOnes = sbase + C::kOnesOff;
      int cnt = 0;  // (q tile, head) pairs, for the Q/dO ring and the S/dP buffer
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int rs = it & 1;
        if (!(ok = mbar_wait(smem_u32(&ring_full[rs]), (it >> 1) & 1, &abort_flag, a.status))) break;
        const WorkItem w = ring[rs];
        mbar_arrive(smem_u32(&ring_taken[rs]));
        mbar_arrive(smem_u32(&ring_empty[rs]));
        if (w.blk < 0) break;
        const int npairs = (w.t1 - w.t0 + 1) * a.group;
        if (!(ok = mbar_wait(smem_u32(&bar_kv_full), it & 1, &abort_flag, a.status))) break;
        tc_fence_after();
        // Pairs are software-pipelined inside an item.  The bf16 P^T and dS^T
        // of pair n go into the dP^T columns (each warpgroup writes them over
        // its own 64 dP^T columns once it has read them), so the S^T columns
        // are free as soon as S^T(n) is in registers:
        //   S^T(0) dP^T(0) | S^T(1) dV(0) dK(0) dP^T(1) | S^T(2) dV(1) dK(1) ...
        // S^T(n+1) runs while the elementwise warps wait for dP^T(n) and
        // compute dS^T(n); their exp2 work of pair n+1 runs during dV(n),
        // dK(n) and dP^T(n+1).  dP^T(n+1) overwrites P^T(n) and dS^T(n) after
        // dV(n) and dK(n) have read them (in-order execution).  Items are not
        // pipelined into each other: the next item's K/V tiles load only once
        // this item's MMAs are done.
        auto issue_s = [&](int c) -> bool {  // S^T of pair c: needs its Q (and staged -lse/scale)
          const int sl = c % S;
          if (!mbar_wait(smem_u32(&bar_qdo_full[sl]), (c / S) & 1, &abort_flag, a.status)) return false;
          tc_fence_after();
          const uint32_t sq = sQ0 + sl * 2 * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::kColS, kmajor_desc(sK, kk), kmajor_desc(sq, kk), idesc_s, kk > 0);
          mma_ss(tmem + C::kColS, aug_desc(sOnes), aug_desc(sbase + C::kQxOff + sl * kAugBytes), idesc_s, 1u);
          tc_commit(smem_u32(&bar_s_full[0]));
          return true;
        };
        auto issue_dp = [&](int c) {  // dP^T of pair c (its Q/dO stage is already waited for)
          const int sl = c % S;
          const uint32_t sdo = sQ0 + sl * 2 * kTileBytes + kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::kColDP, kmajor_desc(sV, kk), kmajor_desc(sdo, kk), idesc_s, kk > 0);
          mma_ss(tmem + C::kColDP, aug_desc(sOnes), aug_desc(sbase + C::kDOxOff + sl * kAugBytes), idesc_s, 1u);
          tc_commit(smem_u32(&bar_s_full[1]));
        };
        // S^T - lse/scale = [K 1] [Q -lse/scale]^T and dP^T - D = [V 1] [dO -D]^T
        // (N = 128 queries; the last k-step is the extra block), committed
        // separately so the exp2 work starts while dP^T runs.
        // K and V are read only by S^T and dP^T: the slot is released once the
        // item's last dP^T is issued (the commit covers every earlier MMA), so
        // the next item's K and V load while this item's last pair finishes.
        if (!(ok = issue_s(cnt))) break;
        issue_dp(cnt);
        if (npairs == 1) tc_commit(smem_u32(&bar_kv_empty));
        for (int pr = 0; pr < npairs && ok; ++pr) {
          const int slot = cnt % S;
          const uint32_t sq = sQ0 + slot * 2 * kTileBytes, sdo = sq + kTileBytes;
          const bool more = pr + 1 < npairs;
          // S^T(n+1) once S^T(n) has been read out, and only if its Q stage
          // has landed: the MMA warp never blocks on that load here (it would
          // hold back dV(n) and dK(n)).
          bool s_next = false;
          if (more) {
            if (!(ok = mbar_wait(smem_u32(&bar_s_free), cnt & 1, &abort_flag, a.status))) break;
            if (mbar_try_wait(smem_u32(&bar_qdo_full[(cnt + 1) % S]), ((cnt + 1) / S) & 1)) {
              tc_fence_after();
              if (!(ok = issue_s(cnt + 1))) break;
              s_next = true;
            }
          }
          // The accumulators of the previous item must have been read out.
          if (pr == 0 && it > 0 &&
              !(ok = mbar_wait(smem_u32(&bar_acc_empty), (it - 1) & 1, &abort_flag, a.status)))
            break;
          // dV += P^T_half dO_half and dK += dS^T_half Q_half as each half
          // arrives (K = 64 queries; P^T in the upper, dS^T in the lower 32
          // of the half's 64 dP^T columns).
          for (int half = 0; half < 2 && ok; ++half) {
            if (!(ok = mbar_wait(smem_u32(&bar_ds_full[half]), cnt & 1, &abort_flag, a.status))) break;
            tc_fence_after();
            const bool acc = pr > 0 || half > 0;
            const uint32_t tdp = tmem + C::kColDP + 64 * half;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tmem + C::kColDV, tdp + 32 + kk * 8, mnmajor_desc(sdo, 4 * half + kk), idesc_g,
                     (acc || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tmem + C::kColDK, tdp + kk * 8, mnmajor_desc(sq, 4 * half + kk), idesc_g,
                     (acc || kk > 0) ? 1u : 0u);
          }
          if (!ok) break;
          tc_commit(smem_u32(&bar_qdo_empty[slot]));
          if (more && !s_next && !(ok = issue_s(cnt + 1))) break;
          if (more) issue_dp(cnt + 1);
          if (pr + 2 == npairs) tc_commit(smem_u32(&bar_kv_empty));
          ++cnt;
        }
        if (!ok) break;
        tc_commit(smem_u32(&bar_acc_full));
      }
    }
  } else if (warp < 4) {
    regs_decrease<104>();
    if (warp == 2 && blockIdx.x == 0) report_long_segments(a);
    if (warp == 3 && lane == 0) {
      // ------------------------------------------------------------ items
      // The next item: claimed from the list, or the next of this CTA's
      // share.  It goes to the other roles through a two-slot ring; an item
      // with blk < 0 tells them there is no more work.  The next claim is
      // made once the MMA thread has started the item before it (one item of
      // look-ahead: the claim's round trip to L2 overlaps that item's work,
      // and a CTA never holds more than one unit it has not started).
      int* cw = claim_words;
      const WorkItem* clist = static_cast<const WorkItem*>(p.unit_lists);
      const int n_units = n_units_s;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        WorkItem w;
        bool have;
        if (cw) {
          const int u = claim_next(cw);
          have = u < n_units;
          if (have) w = claim_item(clist, u);
        } else {
          have = it < nit;
          if (have) w = items[it];
        }
        if (!have) w.blk = -1;
        const int rs = it & 1;
        if (it >= 2 && !(ok = mbar_wait(smem_u32(&ring_empty[rs]), ((it >> 1) - 1) & 1, &abort_flag, a.status)))
          break;
        ring[rs] = w;
        mbar_arrive(smem_u32(&ring_full[rs]));
        if (!have) break;
        if (!(ok = mbar_wait(smem_u32(&ring_taken[rs]), (it >> 1) & 1, &abort_flag, a.status))) break;
      }
    }
  } else {
    // ------------------------------------------------------------ elementwise
    // Warpgroup x = query columns [64x, 64x + 64) of every S^T/dP^T tile;
    // thread = key row.  Its bf16 dS^T and P^T go over its own 64 dP^T
    // columns (dS^T the first 32, P^T the other 32).
    regs_increase<200>();
    const int x = (warp >> 2) - 1;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    const uint32_t tS = lane_base + C::kColS + 64 * x, tDP = lane_base + C::kColDP + 64 * x;
    int cnt = 0;
    uint32_t chain_uses = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int rs = it & 1;
      if (!(ok = mbar_wait_warp(smem_u32(&ring_full[rs]), (it >> 1) & 1, &abort_flag, a.status))) break;
      const WorkItem w = ring[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ring_empty[rs]));
      if (w.blk < 0) break;
      const int k0 = w.seg_lo + w.blk * kTile;
      const int g = w.unit;
      const int j = k0 + row;  // this thread's key token
      for (int b = w.t0; b <= w.t1 && ok; ++b) {
        const int q0 = w.seg_lo + b * kTile + 64 * x;  // first query of this half
        const bool full = tile_fully_visible_kv(k0, w.seg_lo + b * kTile, w.seg_hi, a.window);
        for (int hh = 0; hh < a.group; ++hh) {
          if (!(ok = mbar_wait_warp(smem_u32(&bar_s_full[0]), cnt & 1, &abort_flag, a.status))) break;
          tc_fence_after();
          int c_lo = 0, c_hi = 63;
          if (!full) col_visible_rows(j, q0, w.seg_hi, a.window, c_lo, c_hi);
          // P^T while the dP^T MMA runs: the MMA already subtracted lse/scale,
          // so P = exp2((s - lse/scale) * scale*log2e).  The S^T columns are
          // released as soon as they are in registers.
          // P is kept as the bf16 pairs the dV MMA reads; dS^T is computed
          // from the same rounded values.
          uint32_t pp[32];
          {
            uint32_t sr[64];
            tmem_ld64_wait(tS, sr);
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_s_free));
            const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
#pragma unroll
            for (int cc = 0; cc < 64; cc += 2) {
              float p0, p1;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])), sc2), p0, p1);
              p0 = ex2_approx(p0);
              p1 = ex2_approx(p1);
              if (!full) {
                p0 = (cc >= c_lo && cc <= c_hi) ? p0 : 0.f;
                p1 = (cc + 1 >= c_lo && cc + 1 <= c_hi) ? p1 : 0.f;
              }
              pp[cc / 2] = pack_bf16x2(p0, p1);
            }
          }
          // dS^T = P (dP - D) once dP^T is there (the MMA subtracted D); dS^T
          // (bf16) goes over the first 32 of this half's dP^T columns, P^T
          // over the other 32.
          if (!(ok = mbar_wait_warp(smem_u32(&bar_s_full[1]), cnt & 1, &abort_flag, a.status))) break;
          tc_fence_after();
          {
            uint32_t dr[64];
            tmem_ld64_wait(tDP, dr);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              uint32_t pd[16], ph[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int cc = 32 * hf + 2 * e;
                const uint32_t w2 = pp[16 * hf + e];
                const float q0 = __uint_as_float(w2 << 16), q1 = __uint_as_float(w2 & 0xffff0000u);
                float d0, d1;
                f2_unpack(f2_mul(f2_pack(q0, q1), f2_pack(__uint_as_float(dr[cc]), __uint_as_float(dr[cc + 1]))), d0, d1);
                pd[e] = pack_bf16x2(d0, d1);
                ph[e] = w2;
              }
              tmem_st16(tDP + 16 * hf, pd);
              tmem_st16(tDP + 32 + 16 * hf, ph);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_ds_full[x]));
          }
          ++cnt;
        }
      }
      if (!ok) break;
      // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (x scale).
      if (!(ok = mbar_wait_warp(smem_u32(&bar_acc_full), it & 1, &abort_flag, a.status))) break;
      tc_fence_after();
      const bool valid = j < w.seg_hi && token_in_range(j, a.total);
      const RowStrides dst_st = x == 0 ? p.dv_st : p.dk_st;
      void* dst_row = static_cast<__nv_bfloat16*>(x == 0 ? p.dv : p.dk) + j * dst_st.token + g * dst_st.head;
      const uint32_t tacc = lane_base + (x == 0 ? C::kColDV : C::kColDK);
      const float mul = x == 0 ? 1.f : a.scale;
      if (w.chain < 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tacc + c * 32, r);
          tmem_wait_ld(r);
          store_rows32_bf16(dst_row, dst_st.token * 2, c * 32, r, mul, valid);
        }
      } else {
        // A chunk of a split kv item.  Every chunk writes its fp32 partial sums
        // to a buffer of its own; the warpgroup that arrives last (an atomic
        // count per chain) adds all of them in chunk order and stores the
        // result.  The order of the additions is fixed, so the bits do not
        // depend on which chunk finishes last, and no chunk ever waits for
        // another CTA.
        const int li = link_index(w), lk = link_count(w);
        constexpr size_t kBuf = 128 * 128;
        // Buffer layout [32 groups of 4 columns][128 rows][4]: a warp's 32 rows
        // read or write 512 contiguous bytes per group (coalesced).
        float* chain0 = p.chains + ((size_t)w.chain * 2 + x) * kBuf + (size_t)row * 4;
        float* mine = chain0 + (size_t)li * 2 * kBuf;
        int* arrivals = p.chain_progress + w.chain * 2 + x;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tacc + c * 32, r);
          tmem_wait_ld(r);
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            __stcg(reinterpret_cast<float4*>(mine + ((c * 32 + e) >> 2) * 512),
                   make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                               __uint_as_float(r[e + 3])));
        }
        // Every row of the warpgroup has written its part (each thread fences
        // its own stores first), then one thread counts the arrival.
        __threadfence();
        mbar_arrive(smem_u32(&bar_chain[x]));
        if (!(ok = mbar_wait_warp(smem_u32(&bar_chain[x]), chain_uses & 1, &abort_flag, a.status))) break;
        ++chain_uses;
        if (row == 0) {
          // The last arrival also resets the count (every chunk of the chain
          // has counted by then), so the pass can run again on the same
          // workspace; the preprocess resets it as well.
          const bool last = atomicAdd(arrivals, 1) == lk - 1;
          if (last) atomicExch(arrivals, 0);
          chain_last[x] = last;
        }
        mbar_arrive(smem_u32(&bar_chain[x]));
        if (!(ok = mbar_wait_warp(smem_u32(&bar_chain[x]), chain_uses & 1, &abort_flag, a.status))) break;
        ++chain_uses;
        if (chain_last[x]) {
          // Sum in chunk order, 64 columns at a time: every other chunk's
          // partial comes from L2 (16 loads in flight per thread), this
          // chunk's own from TMEM, where it still is.
          __threadfence();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t acc[64];
            for (int q = 0; q < lk; ++q) {
              uint32_t v[64];
              if (q == li) {
                tmem_ld64_wait(tacc + 64 * half, v);
              } else {
                const float* src = chain0 + (size_t)q * 2 * kBuf + (size_t)(16 * half) * 512;
#pragma unroll
                for (int g = 0; g < 16; ++g) {
                  const float4 f = __ldcg(reinterpret_cast<const float4*>(src + g * 512));
                  v[4 * g + 0] = __float_as_uint(f.x);
                  v[4 * g + 1] = __float_as_uint(f.y);
                  v[4 * g + 2] = __float_as_uint(f.z);
                  v[4 * g + 3] = __float_as_uint(f.w);
                }
              }
#pragma unroll
              for (int e = 0; e < 64; ++e)
                acc[e] = q == 0 ? v[e] : __float_as_uint(__uint_as_float(acc[e]) + __uint_as_float(v[e]));
            }
            store_rows32_bf16(dst_row, dst_st.token * 2, 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&acc[0]), mul,
                              valid);
            store_rows32_bf16(dst_row, dst_st.token * 2, 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&acc[32]),
                              mul, valid);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_acc_empty));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && claim_words) claim_finish(claim_words);
}

// ============================================================== dQ pass
struct DqCfg {
  static constexpr int kKStages = 3;  // K tiles: held from S(c) until dQ(c)
  static constexpr int kVStages = 2;  // V tiles: held only until dP(c)
  static constexpr int kMaxItems = 64;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kDOOff = kTileBytes;
  static constexpr uint32_t kKOff = 2 * kTileBytes;
  static constexpr uint32_t kVOff = kKOff + kKStages * kTileBytes;
  static constexpr uint32_t kStateOff = kVOff + kVStages * kTileBytes;  // 224 KB of tiles, then the state below
  static constexpr uint32_t kTmemCols = 512;
  // S buffers b = 0, 1 at 128b (fp32; bf16 dS over them), dP, dQ.
  static constexpr uint32_t kColDP = 256, kColDQ = 384;
};

// Everything else the dQ kernel keeps in shared memory, carved from the
// dynamic allocation after the tiles (the tiles need all but ~3 KB of it, so
// nothing is declared statically and no alignment slack is spent).
struct DqState {
  WorkItem items[DqCfg::kMaxItems];
  WorkItem ring[2];  // the items in flight, handed from the claiming warp to the other roles
  uint64_t item_full[2], item_taken[2], item_empty[2];
  uint64_t q_full, q_empty;
  uint64_t k_full[DqCfg::kKStages], k_empty[DqCfg::kKStages];
  uint64_t v_full[DqCfg::kVStages], v_empty[DqCfg::kVStages];
  uint64_t s_full[2], p_full[2][2];  // p_full[buffer][half]
  uint64_t dp_full, dp_free, acc_full, acc_empty;
  int n_items;
  int claim_mode;  // units are claimed at run time from the workspace list
  int n_units;     // size of that list
  int* claim_words;  // kept here, not in a register, for the end of the kernel
  uint32_t tmem_slot;
  int abort_flag;
};

constexpr uint32_t kDqSmemBytes = DqCfg::kStateOff + sizeof(DqState);
static_assert(kDqSmemBytes <= 227 * 1024, "the dQ kernel's shared memory fits one CTA per SM");

__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const BwdParams p) {
  using C = DqCfg;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const AttnParams& a = p.a;
  const uint32_t sbase = smem_u32(smem_raw);
  // The swizzled tiles need a 1024-byte-aligned base; there is no static
  // shared memory in this kernel, so the dynamic allocation starts aligned.
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicExch(a.status, kStatusSmemAlign);
    return;
  }
  uint8_t* gbase = smem_raw;
  DqState& st = *reinterpret_cast<DqState*>(smem_raw + C::kStateOff);
  WorkItem* items = st.items;
  const uint32_t sQ = sbase + C::kQOff, sDO = sbase + C::kDOOff, sK = sbase + C::kKOff, sV = sbase + C::kVOff;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_ptr = &st.abort_flag;
#define abort_flag (*abort_ptr)
#define bar_q_full st.q_full
#define bar_q_empty st.q_empty
#define bar_s_full st.s_full
#define bar_p_full st.p_full
#define bar_dp_full st.dp_full
#define bar_dp_free st.dp_free
#define bar_acc_full st.acc_full
#define bar_acc_empty st.acc_empty
#define tmem_slot st.tmem_slot
#define n_items st.n_items

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q_full), 1);
    mbar_init(smem_u32(&bar_q_empty), 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(smem_u32(&st.k_full[s]), 1);
      mbar_init(smem_u32(&st.k_empty[s]), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(smem_u32(&st.v_full[s]), 1);
      mbar_init(smem_u32(&st.v_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bar_s_full[b]), 1);
      mbar_init(smem_u32(&bar_p_full[b][0]), 128);
      mbar_init(smem_u32(&bar_p_full[b][1]), 128);
    }
    mbar_init(smem_u32(&bar_dp_full), 1);
    mbar_init(smem_u32(&bar_dp_free), 256);
    mbar_init(smem_u32(&bar_acc_full), 1);
    mbar_init(smem_u32(&bar_acc_empty), 256);
    for (int r = 0; r < 2; ++r) {
      mbar_init(smem_u32(&st.item_full[r]), 1);
      mbar_init(smem_u32(&st.item_taken[r]), 1);
      mbar_init(smem_u32(&st.item_empty[r]), 10);  // the producer, the MMA thread, the 8 elementwise warps
    }
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
  // Inputs written by earlier kernels are read after this wait.  Right after
  // the dK/dV kernel of the same backward there is nothing to wait for: that
  // kernel only starts this one once all of its CTAs have passed their own
  // wait (so delta and every input are complete), and it writes nothing this
  // kernel reads.
  if (!p.dq_after_dkdv) grid_dependency_wait();
  // Work list: the planning kernel of this backward has written the
  // longest-first list and every CTA claims units at run time (claim.cuh);
  // without a fresh list every CTA plans its own share.
  int* const cw = p.sched ? p.sched + kSchedWords : nullptr;
  WorkItem* const clist = cw ? reinterpret_cast<WorkItem*>(p.unit_lists) + kMaxDynUnits : nullptr;
  if (threadIdx.x == 0) {
    st.claim_mode = cw ? claim_ready(cw) : 0;
    st.n_units = st.claim_mode ? __ldcg(cw + 3) : 0;
    st.claim_words = st.claim_mode ? cw : nullptr;
    n_items = 0;
  }
  __syncthreads();
  const int planned = st.claim_mode ? 0
                                    : plan_schedule<false>(a.cu_seqlens, a.nseg, a.window, a.max_levels, a.hq, 0,
                                                           items, C::kMaxItems, reinterpret_cast<int*>(gbase),
                                                           (int)(C::kStateOff / 4), blockIdx.x, gridDim.x);
  if (planned == kPlanDoesNotFit) {
    if (warp == 3) {
      int* cu = reinterpret_cast<int*>(gbase + C::kKOff);
      for (int s = lane; s <= a.nseg; s += 32) cu[s] = a.cu_seqlens[s];
      __syncwarp();
      const int n = build_schedule<false>(cu, a.nseg, a.window, a.max_levels, a.hq, 0, items, C::kMaxItems,
                                          cu + kMaxSegments + 1, blockIdx.x, gridDim.x);
      if (lane == 0) {
        n_items = n < 0 ? 0 : n;
        if (n < 0) atomicExch(a.status, kStatusListOverflow);
      }
    }
  } else if (threadIdx.x == 0 && !st.claim_mode) {
    n_items = planned < 0 ? 0 : planned;
    if (planned < 0) atomicExch(a.status, kStatusListOverflow);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int nit = n_items;
  const bool claim = st.claim_mode;
  const int n_units = st.n_units;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    regs_decrease<104>();
    if (lane == 0) {
      int kc = 0, vc = 0;  // K and V tiles loaded so far
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int rs = it & 1;
        if (!(ok = mbar_wait(smem_u32(&st.item_full[rs]), (it >> 1) & 1, &abort_flag, a.status))) break;
        const WorkItem w = st.ring[rs];
        mbar_arrive(smem_u32(&st.item_empty[rs]));
        if (w.blk < 0) break;
        const int q0 = w.seg_lo + w.blk * kTile;
        const int n0 = w.t0;
        const int h = w.unit, g = h / a.group;
        if (it > 0 && !(ok = mbar_wait(smem_u32(&bar_q_empty), (it - 1) & 1, &abort_flag, a.status))) break;
        mbar_arrive_expect_tx(smem_u32(&bar_q_full), 2 * kTileBytes);
        tma_load_3d(sQ, &tmQ, smem_u32(&bar_q_full), 0, h, q0);
        tma_load_3d(sQ + kHalfTile, &tmQ, smem_u32(&bar_q_full), 64, h, q0);
        tma_load_3d(sDO, &tmDO, smem_u32(&bar_q_full), 0, h, q0);
        tma_load_3d(sDO + kHalfTile, &tmDO, smem_u32(&bar_q_full), 64, h, q0);
        for (int n = n0; n <= w.t1 && ok; ++n) {
          const int k0 = w.seg_lo + n * kTile;
          {
            const int slot = kc % C::kKStages, use = kc / C::kKStages;
            if (use > 0 && !(ok = mbar_wait(smem_u32(&st.k_empty[slot]), (use - 1) & 1, &abort_flag, a.status)))
              break;
            const uint32_t bar = smem_u32(&st.k_full[slot]);
            mbar_arrive_expect_tx(bar, kTileBytes);
            tma_load_3d(sK + slot * kTileBytes, &tmK, bar, 0, g, k0);
            tma_load_3d(sK + slot * kTileBytes + kHalfTile, &tmK, bar, 64, g, k0);
            ++kc;
          }
          {
            const int slot = vc % C::kVStages, use = vc / C::kVStages;
            if (use > 0 && !(ok = mbar_wait(smem_u32(&st.v_empty[slot]), (use - 1) & 1, &abort_flag, a.status)))
              break;
            const uint32_t bar = smem_u32(&st.v_full[slot]);
            mbar_arrive_expect_tx(bar, kTileBytes);
            tma_load_3d(sV + slot * kTileBytes, &tmV, bar, 0, g, k0);
            tma_load_3d(sV + slot * kTileBytes + kHalfTile, &tmV, bar, 64, g, k0);
            ++vc;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per kv tile c (counted over all items): S(c) into buffer c & 1, dP(c)
    // into the single dP buffer once dP(c-1) has been read, then dQ(c) half
    // by half as the elementwise warpgroups finish.  S(c+1) and dP(c+1) are
    // issued before dQ(c), so they overlap this tile's elementwise work.
    regs_decrease<104>();
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, 0, 0);   // S, dP: 128 queries x 128 keys
      constexpr uint32_t idesc_g = make_idesc_bf16(128, 128, 0, 1);   // dQ: 128 queries x 128 dims
      int c = 0;  // kv tiles issued (S/dP), over all items
      bool ok = true;
      // K(cc) lives in K slot cc % 3, V(cc) in V slot cc % 2.
      auto wait_k = [&](int cc) -> bool {
        if (!mbar_wait(smem_u32(&st.k_full[cc % C::kKStages]), (cc / C::kKStages) & 1, &abort_flag, a.status))
          return false;
        tc_fence_after();
        return true;
      };
      auto issue_s = [&](int cc) {
        const uint32_t kt = sK + (cc % C::kKStages) * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + 128 * (cc & 1), kmajor_desc(sQ, kk), kmajor_desc(kt, kk), idesc_s, kk > 0);
        tc_commit(smem_u32(&bar_s_full[cc & 1]));
      };
      auto issue_dp = [&](int cc) -> bool {
        // dP(cc) overwrites dP(cc-1): wait until both warpgroups have read it.
        if (cc > 0 && !mbar_wait(smem_u32(&bar_dp_free), (cc - 1) & 1, &abort_flag, a.status)) return false;
        if (!mbar_wait(smem_u32(&st.v_full[cc % C::kVStages]), (cc / C::kVStages) & 1, &abort_flag, a.status))
          return false;
        tc_fence_after();
        const uint32_t vt = sV + (cc % C::kVStages) * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + C::kColDP, kmajor_desc(sDO, kk), kmajor_desc(vt, kk), idesc_s, kk > 0);
        tc_commit(smem_u32(&bar_dp_full));
        tc_commit(smem_u32(&st.v_empty[cc % C::kVStages]));  // V(cc) is free once dP(cc) is done
        return true;
      };
      for (int it = 0; ok; ++it) {
        const int rs = it & 1;
        if (!(ok = mbar_wait(smem_u32(&st.item_full[rs]), (it >> 1) & 1, &abort_flag, a.status))) break;
        const WorkItem w = st.ring[rs];
        mbar_arrive(smem_u32(&st.item_taken[rs]));
        mbar_arrive(smem_u32(&st.item_empty[rs]));
        if (w.blk < 0) break;
        const int nt = w.t1 - w.t0 + 1;
        if (!(ok = mbar_wait(smem_u32(&bar_q_full), it & 1, &abort_flag, a.status))) break;
        tc_fence_after();
        // Q and dO are read only by S and dP: their buffer is released once the
        // item's last dP is issued, so the next item's Q and dO load while
        // this item's last tile finishes.
        if (!(ok = wait_k(c))) break;
        issue_s(c);
        if (!(ok = issue_dp(c))) break;
        if (nt == 1) tc_commit(smem_u32(&bar_q_empty));
        for (int n = 0; n < nt && ok; ++n, ++c) {
          if (n + 1 < nt) {
            // Next tile's S, and its dP as soon as this tile's dP has been
            // read, so both are ready when the elementwise work moves on.
            if (!(ok = wait_k(c + 1))) break;
            issue_s(c + 1);
            if (!(ok = issue_dp(c + 1))) break;
            if (n + 2 == nt) tc_commit(smem_u32(&bar_q_empty));
          }
          if (n == 0 && it > 0 && !(ok = mbar_wait(smem_u32(&bar_acc_empty), (it - 1) & 1, &abort_flag, a.status)))
            break;
          const uint32_t kt = sK + (c % C::kKStages) * kTileBytes;
          for (int half = 0; half < 2 && ok; ++half) {
            if (!(ok = mbar_wait(smem_u32(&bar_p_full[c & 1][half]), (c >> 1) & 1, &abort_flag, a.status))) break;
            tc_fence_after();
            // dQ += dS_half K_half: bf16 dS of keys [64 half, +64) over the
            // first 32 columns of that half of S buffer c & 1.
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tmem + C::kColDQ, tmem + 128 * (c & 1) + 64 * half + kk * 8, mnmajor_desc(kt, 4 * half + kk),
                     idesc_g, (n > 0 || half > 0 || kk > 0) ? 1u : 0u);
          }
          if (!ok) break;
          tc_commit(smem_u32(&st.k_empty[c % C::kKStages]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&bar_acc_full));
      }
    }
  } else if (warp < 4) {
    regs_decrease<104>();
    if (warp == 2 && blockIdx.x == 0) report_long_segments(a);
    if (warp == 3 && lane == 0) {
      // ------------------------------------------------------------ items
      // The next item: claimed from the list, or the next of this CTA's
      // share.  It goes to the other roles through a two-slot ring; an item
      // with blk < 0 tells them there is no more work.  The next claim is
      // made once the MMA thread has started the item before it (one item of
      // look-ahead: the claim's round trip to L2 overlaps that item's work,
      // and a CTA never holds more than one unit it has not started).
      bool ok = true;
      for (int it = 0; ok; ++it) {
        WorkItem w;
        bool have;
        if (claim) {
          const int u = claim_next(cw);
          have = u < n_units;
          if (have) w = claim_item(clist, u);
        } else {
          have = it < nit;
          if (have) w = items[it];
        }
        if (!have) w.blk = -1;
        const int rs = it & 1;
        if (it >= 2 && !(ok = mbar_wait(smem_u32(&st.item_empty[rs]), ((it >> 1) - 1) & 1, &abort_flag, a.status)))
          break;
        st.ring[rs] = w;
        mbar_arrive(smem_u32(&st.item_full[rs]));
        if (!have) break;
        if (!(ok = mbar_wait(smem_u32(&st.item_taken[rs]), (it >> 1) & 1, &abort_flag, a.status))) break;
      }
    }
  } else {
    // ------------------------------------------------------------ elementwise
    // Warpgroup x = keys [64x, 64x + 64) of every kv tile; thread = query row.
    regs_increase<200>();
    const int x = (warp >> 2) - 1;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    int c = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int rs = it & 1;
      if (!(ok = mbar_wait_warp(smem_u32(&st.item_full[rs]), (it >> 1) & 1, &abort_flag, a.status))) break;
      const WorkItem w = st.ring[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&st.item_empty[rs]));
      if (w.blk < 0) break;
      const int q0 = w.seg_lo + w.blk * kTile;
      const int h = w.unit;
      const int i = q0 + row;  // this thread's query token
      const bool valid = i < w.seg_hi && token_in_range(i, a.total);
      const float lse2 = valid ? p.lse[(size_t)h * a.total + i] * kLog2e : 0.f;
      const float dlt = valid ? p.delta[(size_t)h * a.total + i] : 0.f;
      const uint64_t nl2 = f2_pack(-lse2, -lse2), nd2 = f2_pack(-dlt, -dlt);
      const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
      for (int n = w.t0; n <= w.t1; ++n, ++c) {
        const int kt0 = w.seg_lo + n * kTile;
        const uint32_t tS = lane_base + 128 * (c & 1) + 64 * x;
        const uint32_t tDP = lane_base + C::kColDP + 64 * x;
        if (!(ok = mbar_wait_warp(smem_u32(&bar_s_full[c & 1]), (c >> 1) & 1, &abort_flag, a.status))) break;
        if (!(ok = mbar_wait_warp(smem_u32(&bar_dp_full), c & 1, &abort_flag, a.status))) break;
        tc_fence_after();
        uint32_t sr[64], dr[64];
        tmem_ld64_wait(tS, sr);
        tmem_ld64_wait(tDP, dr);
        // dP is in registers: let the next tile's dP MMA overwrite it.
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_dp_free));
        int c_lo = 0, c_hi = 63;
        const bool full = tile_fully_visible(q0, kt0, a.window);
        if (!full) row_visible_cols(i, kt0 + 64 * x, a.window, c_lo, c_hi);
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int cc = 2 * e;
          float p0, p1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])), sc2, nl2), p0, p1);
          p0 = ex2_approx(p0);
          p1 = ex2_approx(p1);
          if (!full) {
            p0 = (cc >= c_lo && cc <= c_hi) ? p0 : 0.f;
            p1 = (cc + 1 >= c_lo && cc + 1 <= c_hi) ? p1 : 0.f;
          }
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p0, p1),
                           f2_add(f2_pack(__uint_as_float(dr[cc]), __uint_as_float(dr[cc + 1])), nd2)),
                    d0, d1);
          pk[e] = pack_bf16x2(d0, d1);
        }
        tmem_st32(tS, pk);
        tmem_wait_st();
        tc_fence_before();
        // One barrier per S buffer: a warp that has finished this tile may run
        // on to the next one (its S and dP are issued before this tile's dQ)
        // and arrive again before the slowest warp of its warpgroup arrives
        // here; with a single barrier that early arrival would complete this
        // tile's phase too soon.
        mbar_arrive(smem_u32(&bar_p_full[c & 1][x]));
      }
      if (!ok) break;
      // ---- epilogue: warpgroup x writes dQ columns [64x, 64x + 64) (x scale).
      if (!(ok = mbar_wait_warp(smem_u32(&bar_acc_full), it & 1, &abort_flag, a.status))) break;
      tc_fence_after();
      void* dq_row = static_cast<__nv_bfloat16*>(p.dq) + i * p.dq_st.token + h * p.dq_st.head;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t r[32];
        tmem_ld32(lane_base + C::kColDQ + 64 * x + cc * 32, r);
        tmem_wait_ld(r);
        store_rows32_bf16(dq_row, p.dq_st.token * 2, 64 * x + cc * 32, r, a.scale, valid);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_acc_empty));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && st.claim_words) claim_finish(st.claim_words);
  // Finish no earlier than the kernel before (stream order for what follows).
  grid_dependency_wait();
}

#undef abort_flag
#undef bar_q_full
#undef bar_q_empty
#undef bar_s_full
#undef bar_p_full
#undef bar_dp_full
#undef bar_dp_free
#undef bar_acc_full
#undef bar_acc_empty
#undef tmem_slot
#undef n_items

long long persistent_grid(long long units, int num_sms, int max_items) {
  long long grid = num_sms;
  const long long need = (units + max_items - 1) / max_items;
  if (need > grid) grid = need;
  if (units < grid) grid = units > 0 ? units : 1;
  return grid;
}

long long dkdv_grid(const BwdParams& p, int num_sms) {
  return persistent_grid(upper_bound_tiles(p.a.total, p.a.nseg) * p.a.hkv, num_sms, kBwdMaxItems);
}

// ============================================================== planning
// Two CTAs write the longest-first unit lists to the workspace and set the
// claim words (claim.cuh): CTA 0 the dK/dV pass's (kv tiles, long ones split
// into chunks exactly as the pass itself would split them for its grid),
// CTA 1 the dQ pass's.  Inside a backward they run beside the preprocess:
// they read only cu_seqlens, which is complete once the preprocess has let
// them start, and the grid finishes no earlier than the preprocess, so the
// passes that wait for it also find D complete.
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_plan_kernel(const BwdParams p, int dkdv_ctas, int after_pre, int scratch_ints) {
  extern __shared__ int plan_smem[];
  const AttnParams& a = p.a;
  if (!after_pre) grid_dependency_wait();
  WorkItem* lists = static_cast<WorkItem*>(p.unit_lists);
  if (blockIdx.x == 0) {
    const int n = plan_schedule<true>(a.cu_seqlens, a.nseg, a.window, a.max_levels, a.hkv, p.chains_max, nullptr, 0,
                                      plan_smem, scratch_ints, 0, dkdv_ctas, lists, kMaxDynUnits);
    if (threadIdx.x == 0) claim_init(p.sched, n);
  } else {
    const int n = plan_schedule<false>(a.cu_seqlens, a.nseg, a.window, a.max_levels, a.hq, 0, nullptr, 0,
                                       plan_smem, scratch_ints, 0, 1, lists + kMaxDynUnits, kMaxDynUnits);
    if (threadIdx.x == 0) claim_init(p.sched + kSchedWords, n);
  }
  __syncthreads();
  grid_dependents_launch();
  grid_dependency_wait();
}

}  // namespace

int launch_bwd_plan(const BwdParams& p, int num_sms, int after_pre, cudaStream_t stream) {
  const int ints = plan_scratch_ints(p.a.nseg, 1, kBwdThreads);
  const size_t smem = (size_t)ints * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(bwd_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return (int)launch_pdl(bwd_plan_kernel, dim3(2), dim3(kBwdThreads), smem, stream, p, (int)dkdv_grid(p, num_sms),
                         after_pre, ints);
}

int launch_bwd_dkdv(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmDO,
                    const BwdParams& p, int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)DkvCfg::kSmemBytes);
  if (e != cudaSuccess) return (int)e;
  const long long g = dkdv_grid(p, num_sms);
  return (int)launch_pdl(attn_bwd_dkdv_kernel, dim3((unsigned)g), dim3(kBwdThreads), DkvCfg::kSmemBytes, stream, tmQ,
                         tmK, tmV, tmDO, p);
}

int launch_bwd_dq(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmDO,
                  const BwdParams& p, int num_sms, cudaStream_t stream) {
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDqSmemBytes);
  if (e != cudaSuccess) return (int)e;
  const long long g = persistent_grid(upper_bound_tiles(p.a.total, p.a.nseg) * p.a.hq, num_sms, DqCfg::kMaxItems);
  return (int)launch_pdl(attn_bwd_dq_kernel, dim3((unsigned)g), dim3(kBwdThreads), kDqSmemBytes, stream, tmQ,
                         tmK, tmV, tmDO, p);
}

}  // namespace vsw
