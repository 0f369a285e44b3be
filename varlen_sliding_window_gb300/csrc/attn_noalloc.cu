// Backward without any device allocation.
//
// attn_varlen_bwd takes its scratch (delta = rowsum(dout * out), fp32
// [Hq, T]) from the stream-ordered allocator.  Some callers cannot allocate:
// code that runs under an allocator it does not own (a framework caching
// allocator or a fixed, pre-reserved memory budget), callers in real-time or
// embedded settings where a driver allocation may block or synchronise, and
// code paths that must never call cudaMalloc at all.  attn_varlen_bwd_noalloc
// gives them the same backward with the scratch in a fixed, file-scope device
// array instead.  It calls no cudaMalloc, cudaFree or allocating library
// routine.
//
// The array is kNoAllocMaxDelta floats (8 MiB; T * Hq <= 2,097,152); every
// GPU that loads the library keeps it until the process exits.  It holds D
// first; the rest, if any, serves as the dK/dV pass's chain buffers.  All
// calls on a device share it and it keeps the previous call's contents: the
// preprocess overwrites every element of D and resets the chain counters, so
// nothing needs to start at zero, but calls whose GPU work overlaps (two
// streams, or two host threads) race on it and must be serialised.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn_varlen.h"

namespace {

constexpr long long kNoAllocMaxDelta = 1LL << 21;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_delta[kNoAllocMaxDelta];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// The device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached.
int noalloc_scratch(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return ATTN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_delta) != cudaSuccess || !p) return ATTN_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_varlen_bwd_noalloc(const void* dout, const void* q, const void* k, const void* v,
                                       const void* out, const float* lse, const int32_t* cu_seqlens,
                                       int32_t max_seqlen, int32_t window_left, float softmax_scale, void* dq,
                                       void* dk, void* dv, int64_t total, int32_t num_heads_q,
                                       int32_t num_heads_kv, int32_t head_dim, int32_t num_segments, void* stream) {
  // Argument checks up front, so that a rejected call enqueues nothing.
  const void* ptrs[] = {dout, q, k, v, out, lse, cu_seqlens, dq, dk, dv};
  for (const void* x : ptrs)
    if (!x) return ATTN_ERR_NULL_POINTER;
  for (const void* x : ptrs)
    if (reinterpret_cast<uintptr_t>(x) & 15u) return ATTN_ERR_ALIGNMENT;
  if (total < 0 || num_heads_q <= 0 || num_heads_kv <= 0 || num_segments < 0 || num_heads_q % num_heads_kv != 0 ||
      (total > 0 && num_segments == 0))
    return ATTN_ERR_SHAPE;
  if (head_dim != 128) return ATTN_ERR_HEAD_DIM;
  if (num_heads_q > 1024 || num_segments > 8191) return ATTN_ERR_TOO_LARGE;
  if (window_left < -1) return ATTN_ERR_WINDOW;
  if (!(softmax_scale > 0.f) || softmax_scale > 3.0e38f) return ATTN_ERR_SCALE;
  if (max_seqlen < 0 || (total > 0 && max_seqlen > total)) return ATTN_ERR_MAX_SEQLEN;
  if (total * (long long)num_heads_q > kNoAllocMaxDelta) return ATTN_ERR_NOALLOC_TOO_LARGE;
  if (total == 0) return ATTN_OK;
  float* delta = nullptr;
  int rc = noalloc_scratch(&delta);
  if (rc) return rc;
  // The same three kernels as attn_varlen_bwd, with the fixed scratch.
  // What the array holds beyond D lets the dK/dV pass split long kv tiles.
  const size_t bytes = sizeof(float) * (size_t)kNoAllocMaxDelta;
  rc = attn_varlen_bwd_preprocess(dout, out, delta, bytes, total, num_heads_q, head_dim, stream);
  if (rc) return rc;
  rc = attn_varlen_bwd_dkdv(dout, q, k, v, lse, delta, bytes, cu_seqlens, max_seqlen, window_left, softmax_scale, dk,
                            dv, total, num_heads_q, num_heads_kv, head_dim, num_segments, stream);
  if (rc) return rc;
  return attn_varlen_bwd_dq(dout, q, k, v, lse, delta, bytes, cu_seqlens, max_seqlen, window_left, softmax_scale, dq,
                            total, num_heads_q, num_heads_kv, head_dim, num_segments, stream);
}
