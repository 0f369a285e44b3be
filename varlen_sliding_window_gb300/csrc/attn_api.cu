// C ABI of the library: argument validation, TMA descriptor encoding, scratch
// handling and stream-ordered launches.  See include/attn_varlen.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_internal.h"
#include "attn_varlen.h"
#include "mask.cuh"

namespace vsw {

// Per-device error word written by the kernels (1 = wait timeout, 2 = work
// list overflow).  Host code reaches it through its device address.
__device__ int g_status_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool probed = false;
  bool supported = false;
  int num_sms = 0;
  int* status = nullptr;  // device address of g_status_word
  // Stream-ordered pool for the backward's workspace.  It keeps what it has
  // reserved (release threshold: never), so a synchronisation between steps
  // does not hand the memory back and make the next call map it again.
  cudaMemPool_t pool = nullptr;
  // A caller-registered workspace (attn_varlen_set_workspace): when set,
  // attn_varlen_bwd uses it instead of the pool.
  void* user_ws = nullptr;
  size_t user_ws_bytes = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device(DeviceInfo** info) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.num_sms = sms;
    if (d.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return ATTN_ERR_CUDA;
      d.status = static_cast<int*>(p);
      if (cudaMemset(d.status, 0, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.handleTypes = cudaMemHandleTypeNone;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) return ATTN_ERR_CUDA;
      cuuint64_t keep = ~cuuint64_t(0);
      if (cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess)
        return ATTN_ERR_CUDA;
    }
    d.probed = true;
  }
  if (!d.supported) return ATTN_ERR_DEVICE;
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return ATTN_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *info = &d;
  return ATTN_OK;
}

// [T, heads, 128] bf16 with element strides st -> 3-D map (d, head, token),
// box (64, 1, 128), 128-byte swizzle: one box is a 128-token x 64-column
// swizzled half tile.
int make_tile_map(CUtensorMap* m, const void* base, int heads, int64_t total, const RowStrides& st) {
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)total};
  cuuint64_t strides[2] = {(cuuint64_t)st.head * 2, (cuuint64_t)st.token * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The dense layout [T, heads, 128].
RowStrides contiguous(int heads) { return RowStrides{(long long)heads * 128, 128}; }

// Strides of a [T, heads, 128] view: 16-byte multiples (TMA and 16-byte
// stores), the 128 elements of a (token, head) row never overlap another
// head's row, and a token's heads fit inside one token step.
bool strides_ok(const RowStrides& st, int heads) {
  if (st.token <= 0 || st.head <= 0 || (st.token % 8) != 0 || (st.head % 8) != 0) return false;
  if (st.head < 128 || st.token < st.head * heads) return false;
  return st.token < (1LL << 36);
}

// Reads `n` (token, head) stride pairs from a caller's int64 array.
int read_strides(const int64_t* raw, int n, const int* heads, RowStrides* out) {
  if (!raw) return ATTN_ERR_NULL_POINTER;
  for (int t = 0; t < n; ++t) {
    out[t] = RowStrides{(long long)raw[2 * t], (long long)raw[2 * t + 1]};
    if (!strides_ok(out[t], heads[t])) return ATTN_ERR_STRIDE;
  }
  return ATTN_OK;
}

int validate_common(const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left, float softmax_scale,
                    int64_t total, int32_t hq, int32_t hkv, int32_t head_dim, int32_t nseg) {
  if (!cu_seqlens) return ATTN_ERR_NULL_POINTER;
  if (total < 0 || hq <= 0 || hkv <= 0 || nseg < 0 || (hq % hkv) != 0) return ATTN_ERR_SHAPE;
  if (total > 0 && nseg == 0) return ATTN_ERR_SHAPE;
  if (head_dim != 128) return ATTN_ERR_HEAD_DIM;
  // cu_seqlens is staged in shared memory by every kernel: at most 8191 segments.
  if (total > (int64_t(1) << 30) || hq > 1024 || nseg > kMaxSegments) return ATTN_ERR_TOO_LARGE;
  // Work units (tiles x heads) are numbered with 32-bit integers on the device.
  if (upper_bound_tiles(total, nseg) * hq > (int64_t(1) << 30)) return ATTN_ERR_TOO_LARGE;
  if (window_left < -1) return ATTN_ERR_WINDOW;
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return ATTN_ERR_SCALE;
  if (max_seqlen < 0 || (total > 0 && max_seqlen > total)) return ATTN_ERR_MAX_SEQLEN;
  return ATTN_OK;
}

AttnParams make_params(const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left, float softmax_scale,
                       int64_t total, int32_t hq, int32_t hkv, int32_t nseg, int* status) {
  AttnParams a;
  a.cu_seqlens = cu_seqlens;
  a.nseg = nseg;
  a.total = (int)total;
  a.hq = hq;
  a.hkv = hkv;
  a.group = hq / hkv;
  // A window at least as long as the microbatch is global causal; clamping
  // keeps every index computation far from int overflow.
  a.window = (window_left >= total) ? -1 : window_left;
  a.max_seqlen = max_seqlen;
  a.max_levels = (max_seqlen + kTile - 1) / kTile;
  a.scale = softmax_scale;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.status = status;
  return a;
}

}  // namespace
}  // namespace vsw

using namespace vsw;

namespace {

// st: q, k, v, out.
int fwd_impl(const void* q, const void* k, const void* v, const int32_t* cu_seqlens, int32_t max_seqlen,
             int32_t window_left, float softmax_scale, void* out, float* lse, int64_t total, int32_t num_heads_q,
             int32_t num_heads_kv, int32_t head_dim, int32_t num_segments, const RowStrides* st, void* stream) {
  int rc = validate_common(cu_seqlens, max_seqlen, window_left, softmax_scale, total, num_heads_q, num_heads_kv,
                           head_dim, num_segments);
  if (rc) return rc;
  if (!q || !k || !v || !out || !lse) return ATTN_ERR_NULL_POINTER;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return ATTN_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev))) return rc;
  if (total == 0) return ATTN_OK;
  CUtensorMap tq, tk, tv;
  if (make_tile_map(&tq, q, num_heads_q, total, st[0]) || make_tile_map(&tk, k, num_heads_kv, total, st[1]) ||
      make_tile_map(&tv, v, num_heads_kv, total, st[2]))
    return ATTN_ERR_CUDA;
  FwdParams p;
  p.a = make_params(cu_seqlens, max_seqlen, window_left, softmax_scale, total, num_heads_q, num_heads_kv,
                    num_segments, dev->status);
  p.out = out;
  p.lse = lse;
  p.out_st = st[3];
  if (launch_fwd(tq, tk, tv, p, dev->num_sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_varlen_fwd(const void* q, const void* k, const void* v, const int32_t* cu_seqlens, int32_t max_seqlen,
                    int32_t window_left, float softmax_scale, void* out, float* lse, int64_t total,
                    int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, int32_t num_segments,
                    void* stream) {
  if (num_heads_q <= 0 || num_heads_kv <= 0) return ATTN_ERR_SHAPE;
  const RowStrides st[4] = {contiguous(num_heads_q), contiguous(num_heads_kv), contiguous(num_heads_kv),
                            contiguous(num_heads_q)};
  return fwd_impl(q, k, v, cu_seqlens, max_seqlen, window_left, softmax_scale, out, lse, total, num_heads_q,
                  num_heads_kv, head_dim, num_segments, st, stream);
}

int attn_varlen_fwd_strided(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                            int32_t max_seqlen, int32_t window_left, float softmax_scale, void* out, float* lse,
                            int64_t total, int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim,
                            int32_t num_segments, const int64_t* strides, void* stream) {
  if (num_heads_q <= 0 || num_heads_kv <= 0) return ATTN_ERR_SHAPE;
  const int heads[4] = {num_heads_q, num_heads_kv, num_heads_kv, num_heads_q};
  RowStrides st[4];
  int rc = read_strides(strides, 4, heads, st);
  if (rc) return rc;
  return fwd_impl(q, k, v, cu_seqlens, max_seqlen, window_left, softmax_scale, out, lse, total, num_heads_q,
                  num_heads_kv, head_dim, num_segments, st, stream);
}

size_t attn_varlen_bwd_workspace_bytes(int64_t total, int32_t num_heads_q) {
  if (total <= 0 || num_heads_q <= 0) return 0;
  // delta = rowsum(dout * out), fp32 [Hq, T] (256-byte padded), then the
  // chain counters and buffers that let the dK/dV pass split long kv items.
  return full_workspace_bytes(total, num_heads_q);
}

size_t attn_varlen_workspace_bytes(int64_t total, int32_t num_heads_q, int32_t num_segments, int32_t max_seqlen) {
  // The scratch depends on T and Hq only; the other two are accepted so
  // that a caller can size it from the arguments it passes to the calls.
  if (num_segments < 0 || max_seqlen < 0) return 0;
  return attn_varlen_bwd_workspace_bytes(total, num_heads_q);
}

int attn_varlen_set_workspace(void* dev_ptr, size_t bytes) {
  if (dev_ptr && (reinterpret_cast<uintptr_t>(dev_ptr) & 255u)) return ATTN_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  const int rc = current_device(&dev);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  dev->user_ws = (dev_ptr && bytes) ? dev_ptr : nullptr;
  dev->user_ws_bytes = dev->user_ws ? bytes : 0;
  return ATTN_OK;
}

}  // extern "C"

namespace {

// Validation, device check, tensor maps and parameters shared by the
// backward entry points.
struct BwdSetup {
  DeviceInfo* dev = nullptr;
  CUtensorMap tq, tk, tv, tdo;
  BwdParams p;
};

// st: dout, q, k, v, out, dq, dk, dv (null: all contiguous).
int prepare_bwd(BwdSetup& b, const void* dout, const void* q, const void* k, const void* v, const void* out,
                const float* lse, const void* workspace, const int32_t* cu_seqlens, int32_t max_seqlen,
                int32_t window_left, float softmax_scale, void* dq, void* dk, void* dv, int64_t total,
                int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, int32_t num_segments,
                const RowStrides* st = nullptr) {
  int rc = validate_common(cu_seqlens, max_seqlen, window_left, softmax_scale, total, num_heads_q, num_heads_kv,
                           head_dim, num_segments);
  if (rc) return rc;
  const void* ptrs[] = {dout, q, k, v, lse};
  for (const void* x : ptrs)
    if (!x) return ATTN_ERR_NULL_POINTER;
  for (const void* x : ptrs)
    if (!aligned16(x)) return ATTN_ERR_ALIGNMENT;
  const void* opt[] = {out, workspace, dq, dk, dv};  // the callers pass the ones they need (checked there)
  for (const void* x : opt)
    if (x && !aligned16(x)) return ATTN_ERR_ALIGNMENT;
  if ((rc = current_device(&b.dev))) return rc;
  if (total == 0) return ATTN_OK;
  RowStrides cs[8];
  if (!st) {
    const int heads[8] = {num_heads_q, num_heads_q, num_heads_kv, num_heads_kv,
                          num_heads_q, num_heads_q, num_heads_kv, num_heads_kv};
    for (int t = 0; t < 8; ++t) cs[t] = contiguous(heads[t]);
    st = cs;
  }
  if (make_tile_map(&b.tq, q, num_heads_q, total, st[1]) || make_tile_map(&b.tk, k, num_heads_kv, total, st[2]) ||
      make_tile_map(&b.tv, v, num_heads_kv, total, st[3]) ||
      make_tile_map(&b.tdo, dout, num_heads_q, total, st[0]))
    return ATTN_ERR_CUDA;
  b.p.a = make_params(cu_seqlens, max_seqlen, window_left, softmax_scale, total, num_heads_q, num_heads_kv,
                      num_segments, b.dev->status);
  b.p.dout = dout;
  b.p.out = out;
  b.p.lse = lse;
  b.p.delta = nullptr;
  b.p.chains = nullptr;
  b.p.chain_progress = nullptr;
  b.p.chains_max = 0;
  b.p.sched = nullptr;
  b.p.unit_lists = nullptr;
  b.p.dq_after_dkdv = 0;
  b.p.dq = dq;
  b.p.dk = dk;
  b.p.dv = dv;
  b.p.dout_st = st[0];
  b.p.out_st = st[4];
  b.p.dq_st = st[5];
  b.p.dk_st = st[6];
  b.p.dv_st = st[7];
  return ATTN_OK;
}

}  // namespace

namespace vsw {

int device_for_call(int** status, int* num_sms) {
  DeviceInfo* dev = nullptr;
  const int rc = current_device(&dev);
  if (rc) return rc;
  *status = dev->status;
  *num_sms = dev->num_sms;
  return ATTN_OK;
}

int check_bwd_call(const void* dout, const void* q, const void* k, const void* v, const void* out, const float* lse,
                   const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left, float softmax_scale,
                   const void* dq, const void* dk, const void* dv, int64_t total, int32_t num_heads_q,
                   int32_t num_heads_kv, int32_t head_dim, int32_t num_segments) {
  int rc = validate_common(cu_seqlens, max_seqlen, window_left, softmax_scale, total, num_heads_q, num_heads_kv,
                           head_dim, num_segments);
  if (rc) return rc;
  const void* ptrs[] = {dout, q, k, v, out, lse, dq, dk, dv};
  for (const void* x : ptrs)
    if (!x) return ATTN_ERR_NULL_POINTER;
  for (const void* x : ptrs)
    if (!aligned16(x)) return ATTN_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  return current_device(&dev);
}

int bwd_on_workspace(const void* dout, const void* q, const void* k, const void* v, const void* out,
                     const float* lse, const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left,
                     float softmax_scale, void* dq, void* dk, void* dv, int64_t total, int32_t num_heads_q,
                     int32_t num_heads_kv, int32_t head_dim, int32_t num_segments, const RowStrides* st, void* ws,
                     size_t ws_bytes, void* stream) {
  if (!out || !dq || !dk || !dv) return ATTN_ERR_NULL_POINTER;
  BwdSetup b;
  int rc = prepare_bwd(b, dout, q, k, v, out, lse, nullptr, cu_seqlens, max_seqlen, window_left, softmax_scale, dq,
                       dk, dv, total, num_heads_q, num_heads_kv, head_dim, num_segments, st);
  if (rc || total == 0) return rc;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return ATTN_ERR_ALIGNMENT;
  if (!carve_workspace(ws, ws_bytes, total, num_heads_q, b.p)) return ATTN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Each kernel starts under the tail of the one before: the unit lists of
  // both passes are planned while the preprocess computes D, dQ takes the
  // SMs dK/dV frees.
  int lr = launch_bwd_preprocess(b.p, s);
  if (!lr && b.p.sched) lr = launch_bwd_plan(b.p, b.dev->num_sms, 1, s);
  if (!lr) lr = launch_bwd_dkdv(b.tq, b.tk, b.tv, b.tdo, b.p, b.dev->num_sms, s);
  b.p.dq_after_dkdv = 1;
  if (!lr) lr = launch_bwd_dq(b.tq, b.tk, b.tv, b.tdo, b.p, b.dev->num_sms, s);
  return lr ? ATTN_ERR_CUDA : ATTN_OK;
}

}  // namespace vsw

namespace {

int bwd_impl(const void* dout, const void* q, const void* k, const void* v, const void* out, const float* lse,
             const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left, float softmax_scale, void* dq,
             void* dk, void* dv, int64_t total, int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim,
             int32_t num_segments, const RowStrides* st, void* stream) {
  int rc = check_bwd_call(dout, q, k, v, out, lse, cu_seqlens, max_seqlen, window_left, softmax_scale, dq, dk, dv,
                          total, num_heads_q, num_heads_kv, head_dim, num_segments);
  if (rc || total == 0) return rc;
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev))) return rc;
  void* user_ws = nullptr;
  size_t user_bytes = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    user_ws = dev->user_ws;
    user_bytes = dev->user_ws_bytes;
  }
  if (user_ws)
    return bwd_on_workspace(dout, q, k, v, out, lse, cu_seqlens, max_seqlen, window_left, softmax_scale, dq, dk, dv,
                            total, num_heads_q, num_heads_kv, head_dim, num_segments, st, user_ws, user_bytes, stream);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  const size_t ws_bytes = full_workspace_bytes(total, num_heads_q);
  if (cudaMallocFromPoolAsync(&ws, ws_bytes, dev->pool, s) != cudaSuccess) return ATTN_ERR_ALLOC;
  rc = bwd_on_workspace(dout, q, k, v, out, lse, cu_seqlens, max_seqlen, window_left, softmax_scale, dq, dk, dv, total,
                        num_heads_q, num_heads_kv, head_dim, num_segments, st, ws, ws_bytes, stream);
  const cudaError_t fr = cudaFreeAsync(ws, s);
  if (rc) return rc;
  return fr == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

int attn_varlen_bwd(const void* dout, const void* q, const void* k, const void* v, const void* out,
                    const float* lse, const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left,
                    float softmax_scale, void* dq, void* dk, void* dv, int64_t total, int32_t num_heads_q,
                    int32_t num_heads_kv, int32_t head_dim, int32_t num_segments, void* stream) {
  return bwd_impl(dout, q, k, v, out, lse, cu_seqlens, max_seqlen, window_left, softmax_scale, dq, dk, dv, total,
                  num_heads_q, num_heads_kv, head_dim, num_segments, nullptr, stream);
}

int attn_varlen_bwd_strided(const void* dout, const void* q, const void* k, const void* v, const void* out,
                            const float* lse, const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left,
                            float softmax_scale, void* dq, void* dk, void* dv, int64_t total, int32_t num_heads_q,
                            int32_t num_heads_kv, int32_t head_dim, int32_t num_segments, const int64_t* strides,
                            void* stream) {
  if (num_heads_q <= 0 || num_heads_kv <= 0) return ATTN_ERR_SHAPE;
  const int heads[8] = {num_heads_q, num_heads_q, num_heads_kv, num_heads_kv,
                        num_heads_q, num_heads_q, num_heads_kv, num_heads_kv};
  RowStrides st[8];
  int rc = read_strides(strides, 8, heads, st);
  if (rc) return rc;
  return bwd_impl(dout, q, k, v, out, lse, cu_seqlens, max_seqlen, window_left, softmax_scale, dq, dk, dv, total,
                  num_heads_q, num_heads_kv, head_dim, num_segments, st, stream);
}

int attn_varlen_bwd_preprocess(const void* dout, const void* out, void* workspace, size_t workspace_bytes,
                               int64_t total, int32_t num_heads_q, int32_t head_dim, void* stream) {
  if (!dout || !out || !workspace) return ATTN_ERR_NULL_POINTER;
  if (total < 0 || num_heads_q <= 0) return ATTN_ERR_SHAPE;
  if (head_dim != 128) return ATTN_ERR_HEAD_DIM;
  if (total > (int64_t(1) << 30) || num_heads_q > 1024) return ATTN_ERR_TOO_LARGE;
  if (!aligned16(dout) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  int rc = current_device(&dev);
  if (rc || total == 0) return rc;
  BwdParams p{};
  p.a.total = (int)total;
  p.a.hq = num_heads_q;
  p.dout = dout;
  p.out = out;
  p.dout_st = p.out_st = contiguous(num_heads_q);
  if (!carve_workspace(workspace, workspace_bytes, total, num_heads_q, p)) return ATTN_ERR_WORKSPACE;
  return launch_bwd_preprocess(p, static_cast<cudaStream_t>(stream)) ? ATTN_ERR_CUDA : ATTN_OK;
}

int attn_varlen_bwd_plan(const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left, void* workspace,
                         size_t workspace_bytes, int64_t total, int32_t num_heads_q, int32_t num_heads_kv,
                         int32_t num_segments, void* stream) {
  int rc = validate_common(cu_seqlens, max_seqlen, window_left, 1.f, total, num_heads_q, num_heads_kv, 128,
                           num_segments);
  if (rc) return rc;
  if (!workspace) return ATTN_ERR_NULL_POINTER;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev))) return rc;
  if (total == 0) return ATTN_OK;
  BwdParams p{};
  p.a = make_params(cu_seqlens, max_seqlen, window_left, 1.f, total, num_heads_q, num_heads_kv, num_segments,
                    dev->status);
  if (!carve_workspace(workspace, workspace_bytes, total, num_heads_q, p)) return ATTN_ERR_WORKSPACE;
  // Without room for the lists the passes plan their own shares: nothing to do.
  if (!p.sched) return ATTN_OK;
  return launch_bwd_plan(p, dev->num_sms, 0, static_cast<cudaStream_t>(stream)) ? ATTN_ERR_CUDA : ATTN_OK;
}

int attn_varlen_bwd_dkdv(const void* dout, const void* q, const void* k, const void* v, const float* lse,
                         const void* workspace, size_t workspace_bytes, const int32_t* cu_seqlens, int32_t max_seqlen,
                         int32_t window_left, float softmax_scale, void* dk, void* dv, int64_t total,
                         int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, int32_t num_segments,
                         void* stream) {
  if (!workspace || !dk || !dv) return ATTN_ERR_NULL_POINTER;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_ALIGNMENT;
  BwdSetup b;
  int rc = prepare_bwd(b, dout, q, k, v, nullptr, lse, workspace, cu_seqlens, max_seqlen, window_left, softmax_scale,
                       nullptr, dk, dv, total, num_heads_q, num_heads_kv, head_dim, num_segments);
  if (rc || total == 0) return rc;
  if (!carve_workspace(const_cast<void*>(workspace), workspace_bytes, total, num_heads_q, b.p))
    return ATTN_ERR_WORKSPACE;
  return launch_bwd_dkdv(b.tq, b.tk, b.tv, b.tdo, b.p, b.dev->num_sms, static_cast<cudaStream_t>(stream))
             ? ATTN_ERR_CUDA
             : ATTN_OK;
}

int attn_varlen_bwd_dq(const void* dout, const void* q, const void* k, const void* v, const float* lse,
                       const void* workspace, size_t workspace_bytes, const int32_t* cu_seqlens, int32_t max_seqlen,
                       int32_t window_left, float softmax_scale, void* dq, int64_t total, int32_t num_heads_q,
                       int32_t num_heads_kv, int32_t head_dim, int32_t num_segments, void* stream) {
  if (!workspace || !dq) return ATTN_ERR_NULL_POINTER;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_ALIGNMENT;
  BwdSetup b;
  int rc = prepare_bwd(b, dout, q, k, v, nullptr, lse, workspace, cu_seqlens, max_seqlen, window_left, softmax_scale,
                       dq, nullptr, nullptr, total, num_heads_q, num_heads_kv, head_dim, num_segments);
  if (rc || total == 0) return rc;
  if (!carve_workspace(const_cast<void*>(workspace), workspace_bytes, total, num_heads_q, b.p))
    return ATTN_ERR_WORKSPACE;
  return launch_bwd_dq(b.tq, b.tk, b.tv, b.tdo, b.p, b.dev->num_sms, static_cast<cudaStream_t>(stream))
             ? ATTN_ERR_CUDA
             : ATTN_OK;
}

int attn_varlen_get_status(void* stream, int32_t* device_code) {
  DeviceInfo* dev = nullptr;
  int rc = current_device(&dev);
  if (rc) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaMemset(dev->status, 0, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (device_code) *device_code = word;
  return word ? ATTN_ERR_DEVICE_STATUS : ATTN_OK;
}

const char* attn_varlen_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL_POINTER: return "a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "invalid shape (T, head counts, Hq % Hkv, or segment count)";
    case ATTN_ERR_HEAD_DIM: return "head_dim must be 128";
    case ATTN_ERR_ALIGNMENT: return "a tensor pointer is not 16-byte aligned";
    case ATTN_ERR_WINDOW: return "window_left must be -1 (global) or >= 0";
    case ATTN_ERR_SCALE: return "softmax_scale must be finite and positive";
    case ATTN_ERR_MAX_SEQLEN: return "max_seqlen must be in [0, T]";
    case ATTN_ERR_DEVICE: return "the current device is not an sm_103 (GB300) GPU";
    case ATTN_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case ATTN_ERR_TOO_LARGE: return "problem size beyond the supported range";
    case ATTN_ERR_ALLOC: return "backward scratch allocation failed";
    case ATTN_ERR_DEVICE_STATUS: return "a kernel recorded a device-side error";
    case ATTN_ERR_WORKSPACE: return "workspace smaller than delta (T * Hq floats, 256-byte padded)";
    case ATTN_ERR_STRIDE:
      return "a stride is not a positive multiple of 8 elements, a head step is below 128, or a token step "
             "is below head step x heads";
    case ATTN_ERR_NOALLOC_TOO_LARGE:
      return "T * Hq exceeds the fixed scratch of attn_varlen_bwd_noalloc (2,097,152 floats)";
    default: return "unknown error code";
  }
}

int attn_varlen_mask_ranges(const int32_t* cu_seqlens, int32_t num_segments, int64_t total, int32_t max_seqlen,
                            int32_t window_left, int32_t by_key, int32_t* ranges, void* stream) {
  int rc = validate_common(cu_seqlens, max_seqlen, window_left, 1.f, total, 1, 1, 128, num_segments);
  if (rc) return rc;
  if (!ranges) return ATTN_ERR_NULL_POINTER;
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev))) return rc;
  if (total == 0) return ATTN_OK;
  if (window_left >= total) window_left = -1;
  if (launch_mask_probe(cu_seqlens, num_segments, (int)total, window_left, (max_seqlen + kTile - 1) / kTile,
                        by_key, ranges, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // extern "C"
