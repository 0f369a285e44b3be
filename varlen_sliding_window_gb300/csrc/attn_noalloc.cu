// Backward without any device allocation.
//
// attn_varlen_bwd takes its scratch (delta = rowsum(dout * out), fp32
// [Hq, T], and the dK/dV pass's chain buffers) from the stream-ordered
// allocator.  Some callers cannot allocate: code that runs under an allocator
// it does not own (a framework caching allocator or a fixed, pre-reserved
// memory budget), callers in real-time or embedded settings where a driver
// allocation may block or synchronise, and code paths that must never call
// cudaMalloc at all.  attn_varlen_bwd_noalloc gives them the same backward
// with the scratch in a fixed, file-scope device array instead.  It calls no
// cudaMalloc, cudaFree or allocating library routine.
//
// The array holds kNoAllocMaxDelta floats of delta (8 MiB: T * Hq <=
// 2,097,152), the counters and work lists of the two passes, and as many
// chain buffers as the allocating path uses (320 x 128 KiB), about 50 MiB in
// all; every GPU that loads the library keeps it until the process exits.
// With the same number of chain buffers the dK/dV pass splits its work
// exactly as in attn_varlen_bwd, so the two calls give the same bits.  All calls on a device
// share the array and it keeps the previous call's contents: the preprocess
// overwrites every element of delta and resets the chain counters, so nothing
// needs to start at zero, but calls whose GPU work overlaps (two streams, or
// two host threads) race on it and must be serialised by the caller.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn_internal.h"
#include "attn_varlen.h"

namespace {

constexpr long long kNoAllocMaxDelta = 1LL << 21;
constexpr int kNoAllocMaxDevices = 64;
constexpr size_t kNoAllocBytes = vsw::kProgressBytes + vsw::kListBytes + vsw::kMaxChains * vsw::kChainBytes +
                                 sizeof(float) * (size_t)kNoAllocMaxDelta;
static_assert(kNoAllocBytes % 256 == 0, "the scratch is carved in 256-byte steps");

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocBytes / sizeof(float)];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// The device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached.
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return ATTN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
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
  // The same argument and device checks as attn_varlen_bwd, before anything
  // else, so that a rejected call enqueues nothing and touches no symbol.
  int rc = vsw::check_bwd_call(dout, q, k, v, out, lse, cu_seqlens, max_seqlen, window_left, softmax_scale, dq, dk,
                               dv, total, num_heads_q, num_heads_kv, head_dim, num_segments);
  if (rc) return rc;
  if (total * (long long)num_heads_q > kNoAllocMaxDelta) return ATTN_ERR_NOALLOC_TOO_LARGE;
  if (total == 0) return ATTN_OK;
  void* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;
  // The same launch chain as attn_varlen_bwd, on the fixed scratch.
  return vsw::bwd_on_workspace(dout, q, k, v, out, lse, cu_seqlens, max_seqlen, window_left, softmax_scale, dq, dk,
                               dv, total, num_heads_q, num_heads_kv, head_dim, num_segments, nullptr, scratch,
                               kNoAllocBytes, stream);
}
