// Host/device parameter blocks and launcher declarations shared by the
// translation units of the library.  Not part of the public C ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

namespace vsw {

// Parameters common to every attention kernel.
struct AttnParams {
  const int* cu_seqlens;  // device, [nseg + 1]
  int nseg;
  int total;       // tokens T
  int hq;          // query heads
  int hkv;         // key/value heads
  int group;       // hq / hkv
  int window;      // window_left, -1 = global
  int max_seqlen;  // the caller's bound on every segment length
  int max_levels;  // ceil(max_seqlen / 128)
  float scale;        // softmax_scale
  float scale_log2;   // softmax_scale * log2(e)
  int* status;        // device status word
};

// Element strides of a [T, H, 128] bf16 tensor whose last dimension is
// contiguous: token t, head h starts at t * token + h * head.
struct RowStrides {
  long long token;
  long long head;
};

struct FwdParams {
  AttnParams a;
  void* out;   // bf16 [T, hq, 128]
  float* lse;  // fp32 [hq, T]
  RowStrides out_st;
};

struct BwdParams {
  AttnParams a;
  const void* dout;  // bf16 [T, hq, 128]
  const void* out;   // bf16 [T, hq, 128]
  const float* lse;  // fp32 [hq, T]
  float* delta;      // fp32 [hq, T], scratch: rowsum(dout * out)
  void* dq;          // bf16 [T, hq, 128]
  void* dk;          // bf16 [T, hkv, 128]
  void* dv;          // bf16 [T, hkv, 128]
  // dK/dV chains (split kv items, one partial-sum buffer per chunk), scratch:
  float* chains;         // fp32 [chains_max][2][128][128] partial dV, dK
  int* chain_progress;   // int [chains_max][2] arrival counts, then the scheduling words
  int chains_max;        // 0 disables splitting
  // Run-time work claiming (null: every CTA deals itself a fixed share):
  // kSchedWords ints per pass (dK/dV first, then dQ) and a unit list of
  // kMaxDynUnits work items per pass.
  int* sched;
  void* unit_lists;
  // Set when the dQ kernel is launched right after the dK/dV kernel of the
  // same backward: it then needs nothing that kernel writes, starts on the
  // SMs the dK/dV kernel frees and waits for it only before exiting.
  int dq_after_dkdv;
  RowStrides dout_st, out_st, dq_st, dk_st, dv_st;
};

// Backward workspace layout: delta, the counter area (chain arrival counts,
// then the scheduling words of the two passes), the two unit lists, the chain
// buffers.
constexpr int kMaxChains = 320;
constexpr size_t kChainBytes = 2ull * 128 * 128 * sizeof(float);
constexpr size_t kProgressBytes = 2816;  // kMaxChains * 2 ints, then the scheduling words; 256-byte multiple
constexpr int kSchedWordsOffset = 2 * kMaxChains;  // ints into the counter area
constexpr int kSchedWords = 4;  // per pass: state, next unit, CTAs done, number of units
constexpr int kProgressInts = (int)(kProgressBytes / 4);
static_assert(kSchedWordsOffset + 2 * kSchedWords <= kProgressInts, "scheduling words fit the counter area");
constexpr int kMaxDynUnits = 32768;   // units a pass may claim at run time
constexpr size_t kWorkItemBytes = 36;  // sizeof(WorkItem), checked where the type is defined
constexpr size_t kListBytes = 2ull * kMaxDynUnits * kWorkItemBytes;
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline size_t delta_bytes(long long total, int hq) { return align256((size_t)total * hq * sizeof(float)); }
inline size_t full_workspace_bytes(long long total, int hq) {
  return delta_bytes(total, hq) + kProgressBytes + kListBytes + kMaxChains * kChainBytes;
}
// Carves a caller-provided workspace; returns false if it cannot hold delta.
// Run-time claiming needs the counter area and the lists; splitting long kv
// items needs chain buffers on top.
inline bool carve_workspace(void* ws, size_t bytes, long long total, int hq, BwdParams& p) {
  const size_t db = delta_bytes(total, hq);
  if (!ws || bytes < db) return false;
  char* base = static_cast<char*>(ws);
  p.delta = reinterpret_cast<float*>(base);
  p.chains_max = 0;
  p.chain_progress = nullptr;
  p.chains = nullptr;
  p.sched = nullptr;
  p.unit_lists = nullptr;
  if (bytes >= db + kProgressBytes + kListBytes) {
    p.chain_progress = reinterpret_cast<int*>(base + db);
    p.sched = p.chain_progress + kSchedWordsOffset;
    p.unit_lists = base + db + kProgressBytes;
    const size_t n = (bytes - db - kProgressBytes - kListBytes) / kChainBytes;
    p.chains_max = (int)(n < (size_t)kMaxChains ? n : (size_t)kMaxChains);
    p.chains = reinterpret_cast<float*>(base + db + kProgressBytes + kListBytes);
  }
  return true;
}

// Launchers (return a cudaError_t value).
int launch_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const FwdParams& p,
               int num_sms, cudaStream_t stream);
int launch_bwd_dkdv(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmDO,
                    const BwdParams& p, int num_sms, cudaStream_t stream);
int launch_bwd_dq(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmDO,
                  const BwdParams& p, int num_sms, cudaStream_t stream);
int launch_bwd_preprocess(const BwdParams& p, cudaStream_t stream);
// after_pre: launched right after the preprocess of the same backward (reads
// cu_seqlens before waiting for it).
int launch_bwd_plan(const BwdParams& p, int num_sms, int after_pre, cudaStream_t stream);
int launch_mask_probe(const int* cu_seqlens, int nseg, int total, int window, int max_levels, int by_key,
                      int* ranges, cudaStream_t stream);

// Launches `kernel` on `stream` with programmatic stream serialization, so
// that its CTAs may start (and run their prologue) while the previous kernel
// in the stream drains.  Every kernel of this library calls
// grid_dependency_wait() before reading global memory written earlier, except
// the dQ kernel launched right after the dK/dV kernel of the same backward,
// which reads nothing that kernel writes and waits only before exiting.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Units of work (tile x head unit) an upper bound: used to size grids.
inline long long upper_bound_tiles(long long total, int nseg) { return total / 128 + nseg + 1; }

// Device status words (see attn_varlen_get_status).
enum : int {
  kStatusTimeout = 1,        // a bounded wait gave up
  kStatusListOverflow = 2,   // a CTA's work list did not fit
  kStatusSmemAlign = 3,      // dynamic shared memory not 1024-byte aligned
  kStatusSegmentTooLong = 4, // a segment longer than max_seqlen (its tiles past max_seqlen were skipped)
  kStatusGateRange = 5,      // Kimi Delta: a log decay g at or below -5.8 (or NaN)
};

// Run by one warp: reports, through the status word, a segment longer than
// the caller's max_seqlen.  The kernels' work lists only reach max_seqlen
// (rounded up to a whole tile), so such a segment's later rows are not
// computed; the call itself cannot see cu_seqlens, which lives on the device.
__device__ __forceinline__ void report_long_segments(const AttnParams& a) {
  const int lane = threadIdx.x & 31;
  bool bad = false;
  for (int s = lane; s < a.nseg; s += 32) bad |= (a.cu_seqlens[s + 1] - a.cu_seqlens[s]) > a.max_seqlen;
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicExch(a.status, kStatusSegmentTooLong);
}

// The whole backward (preprocess, dK/dV pass, dQ pass, each kernel starting
// under the tail of the one before) on a caller-provided workspace of
// ws_bytes bytes (256-byte aligned, at least delta_bytes(total, hq)).  st:
// dout, q, k, v, out, dq, dk, dv (null: all dense).  Validates everything
// itself; returns an ATTN_* code.
int bwd_on_workspace(const void* dout, const void* q, const void* k, const void* v, const void* out,
                     const float* lse, const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left,
                     float softmax_scale, void* dq, void* dk, void* dv, int64_t total, int32_t num_heads_q,
                     int32_t num_heads_kv, int32_t head_dim, int32_t num_segments, const RowStrides* st, void* ws,
                     size_t ws_bytes, void* stream);

// The current device's status word and SM count, after the same device
// checks every entry point makes (an sm_103 GPU); returns an ATTN_* code.
int device_for_call(int** status, int* num_sms);

// Argument and device checks shared by the backward entry points, in the
// order every entry point applies them (arguments first, then the device).
int check_bwd_call(const void* dout, const void* q, const void* k, const void* v, const void* out, const float* lse,
                   const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left, float softmax_scale,
                   const void* dq, const void* dk, const void* dv, int64_t total, int32_t num_heads_q,
                   int32_t num_heads_kv, int32_t head_dim, int32_t num_segments);

}  // namespace vsw
