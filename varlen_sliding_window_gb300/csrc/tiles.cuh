// Shared-memory tile geometry shared by the attention kernels.
//
// A 128 x 128 bf16 tile (128 tokens x head dim 128) is stored as two halves
// of 128 rows x 64 columns; each half is the 128-byte-swizzled layout that a
// TMA box of (64, 1, 128) writes and that tcgen05 smem descriptors with
// SWIZZLE_128B read: row r at byte r*128, 16-byte chunk c stored at chunk
// c ^ (r % 8).
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace vsw {

constexpr uint32_t kTileBytes = 128 * 128 * 2;
constexpr uint32_t kHalfTile = kTileBytes / 2;

// K-major operand (rows x 128 K columns), advanced to MMA k-step kk
// (16 columns = 32 bytes inside a swizzled row).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
  return make_sdesc_sw128(tile + (kk >> 2) * kHalfTile + (kk & 3) * 32, 16, 1024);
}

// MN-major B operand stored [K rows][128 N columns], advanced to k-step kk
// (16 rows).  LBO = distance between the two 64-column halves (N direction),
// SBO = distance between 8-row groups (K direction).
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
  return make_sdesc_sw128(tile + kk * 16 * 128, kHalfTile, 1024);
}

// Writes fp32 columns [c, c + 32) of the warp's 32 rows (one row per lane,
// lane l's row at dst_row; consecutive lanes hold consecutive tokens,
// row_stride_bytes apart), times mul, as bf16.  Each quad of lanes first
// swaps 16-byte pieces (a 4 x 4 transpose in two shuffle rounds), so that a
// store instruction writes 64 contiguous bytes of each of 8 rows rather
// than 16 bytes of each of 32 rows: a quarter of the cache lines per
// instruction.  All 32 lanes call it; rows with valid == false are skipped.
__device__ __forceinline__ void store_rows32_bf16(void* dst_row, long long row_stride_bytes, int c,
                                                  const uint32_t (&r)[32], float mul, bool valid) {
  const int lane = threadIdx.x & 31, qi = lane & 3;
  const unsigned vmask = __ballot_sync(0xffffffffu, valid);
  uint32_t x[4][4];  // x[v][k]: word v of 16-byte piece k of this lane's row
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int v = 0; v < 4; ++v)
      x[v][k] = pack_bf16x2(__uint_as_float(r[8 * k + 2 * v]) * mul, __uint_as_float(r[8 * k + 2 * v + 1]) * mul);
  // Round 1 (lane bit 0), round 2 (lane bit 1): a lane keeps the pieces whose
  // index bit equals its own lane bit and trades the others with its partner.
  // Afterwards piece k of lane qi is piece qi of quad lane k's row.
  const bool odd = qi & 1, high = qi & 2;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? x[v][2 * b] : x[v][2 * b + 1], 1);
      if (odd)
        x[v][2 * b] = got;
      else
        x[v][2 * b + 1] = got;
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint32_t got = __shfl_xor_sync(0xffffffffu, high ? x[v][b] : x[v][b + 2], 2);
      if (high)
        x[v][b] = got;
      else
        x[v][b + 2] = got;
    }
  }
  char* mine = static_cast<char*>(dst_row) + 2 * (c + 8 * qi);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if ((vmask >> ((lane & ~3) + k)) & 1u)
      *reinterpret_cast<uint4*>(mine + (long long)(k - qi) * row_stride_bytes) =
          make_uint4(x[0][k], x[1][k], x[2][k], x[3][k]);
}

// One extra k-step of 16 columns appended to a K-major operand: 128 rows x
// 16 bf16 (32 bytes per row) with the 32-byte swizzle, 8-row groups 256 bytes
// apart.  Used to fold a per-row term into an MMA (row x 1 + term x 1).
constexpr uint32_t kAugBytes = 128 * 32;
__device__ __forceinline__ uint64_t aug_desc(uint32_t block) { return make_sdesc_sw32(block, 16, 256); }
// Byte address of the first 16-byte chunk (columns 0..7) of `row`: under the
// 32-byte swizzle the two chunks of a row swap places when bit 2 of the row is set.
__device__ __forceinline__ uint32_t aug_chunk0(uint32_t block, int row) {
  return block + row * 32 + (((uint32_t(row) >> 2) & 1u) << 4);
}

// Byte address of the 16-byte chunk holding columns 8*c8 .. 8*c8+7 of `row`.
__device__ __forceinline__ uint32_t swizzled_chunk(uint32_t tile, int row, int c8) {
  return tile + (c8 >> 3) * kHalfTile + row * 128 + ((uint32_t(c8 & 7) ^ uint32_t(row & 7)) << 4);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace vsw
