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
