/*
 * attn_varlen.h -- C ABI of a GB300 (sm_103a) library for the training-step
 * forward and backward of document-masked causal grouped-query attention.
 *
 * The operation (research.dws.rip/llm/kernels, section 01 "How it was
 * measured", Fig. 2 "Benchmark setup", section 02): a microbatch of T tokens
 * is packed from many documents and cut into rows at the context length.  No
 * token attends across its document boundary or row cut, so attention is
 * confined to segments [cu_seqlens[s], cu_seqlens[s+1]).  Inside a segment it
 * is causal; a local layer additionally limits each query to a left window.
 * Heads are grouped: Hq query heads share Hkv key/value heads (8 and 2 of
 * width 128 on the page), query head h reading kv head h / (Hq / Hkv).
 *
 * Definition, for a query i in segment [a, b) and query head h (g = its kv
 * head):
 *     V(i)   = { j : a <= j <= i  and  (window_left < 0 or i - j <= window_left) }
 *     s_ij   = softmax_scale * <q[i,h,:], k[j,g,:]>
 *     lse[h,i] = log sum_{j in V(i)} exp(s_ij)            (natural log)
 *     out[i,h,:] = sum_{j in V(i)} exp(s_ij - lse[h,i]) * v[j,g,:]
 * The backward returns dq, dk, dv of  L = sum(dout * out).
 * window_left = w keeps w+1 keys including the query itself (a 512-token
 * window is window_left = 512); window_left = -1 is global causal.
 *
 * Layouts (all row-major, contiguous, bf16 = IEEE bfloat16 bit patterns):
 *     q, out, dout, dq : [T, Hq, 128]      k, v, dk, dv : [T, Hkv, 128]
 *     lse              : float32 [Hq, T]
 *     cu_seqlens       : int32 [num_segments + 1], non-decreasing,
 *                        cu_seqlens[0] = 0, cu_seqlens[num_segments] = T.
 * Repeated entries (empty segments) are allowed and change no output bit;
 * they let callers pad the boundary list to a fixed size for CUDA-graph
 * replay (section 06 of the same page).
 *
 * Ownership and memory: every pointer except `stream` is caller-owned DEVICE
 * memory on the current CUDA device, 16-byte aligned.  The library keeps no
 * reference after the enqueued work completes.  Outputs are fully
 * overwritten.  The forward allocates nothing.  attn_varlen_bwd takes a
 * scratch buffer of attn_varlen_bwd_workspace_bytes() bytes, stream-ordered
 * on `stream`, from a per-device memory pool the library creates on its first
 * call on that device (make that first call outside any stream capture); the
 * pool keeps the memory it has reserved for later calls.  A caller that owns
 * its scratch registers it once with attn_varlen_set_workspace(); the
 * backward then uses that buffer and allocates nothing.  The sub-step calls
 * below take a caller-provided workspace as an argument.
 *
 * Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 * stream).  No call synchronises the host except attn_varlen_get_status();
 * all device work is enqueued on `stream`.
 *
 * Errors: every call returns ATTN_OK (0) or a negative ATTN_ERR_* code and
 * never throws.  Argument errors are detected before anything is enqueued.
 * cu_seqlens is only read on the device; a list that breaks the rules above
 * gives unspecified outputs but every loop stays bounded.  Asynchronous device
 * errors are recorded in a per-device status word read by
 * attn_varlen_get_status(): a bounded wait that gave up, a work list that did
 * not fit, or a segment longer than max_seqlen (the kernels compute rows only
 * up to max_seqlen, rounded up to a multiple of 128, so the later rows of such
 * a segment are left unwritten).
 */
#ifndef ATTN_VARLEN_H_
#define ATTN_VARLEN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_OK 0
#define ATTN_ERR_NULL_POINTER (-1)   /* a required pointer is NULL */
#define ATTN_ERR_SHAPE (-2)          /* T < 0, heads <= 0, Hq % Hkv != 0, num_segments < 0 ... */
#define ATTN_ERR_HEAD_DIM (-3)       /* head_dim != 128 */
#define ATTN_ERR_ALIGNMENT (-4)      /* a tensor pointer is not 16-byte aligned */
#define ATTN_ERR_WINDOW (-5)         /* window_left < -1 */
#define ATTN_ERR_SCALE (-6)          /* softmax_scale not finite and > 0 */
#define ATTN_ERR_MAX_SEQLEN (-7)     /* max_seqlen < 0, or > T when T > 0 */
#define ATTN_ERR_DEVICE (-8)         /* current device is not an sm_103 GPU */
#define ATTN_ERR_CUDA (-9)           /* a CUDA runtime/driver call failed */
#define ATTN_ERR_TOO_LARGE (-10)     /* T or a head count beyond the supported range */
#define ATTN_ERR_ALLOC (-11)         /* the backward scratch could not be allocated */
#define ATTN_ERR_DEVICE_STATUS (-12) /* attn_varlen_get_status: a kernel reported an error */
#define ATTN_ERR_NOALLOC_TOO_LARGE (-13) /* attn_varlen_bwd_noalloc: T * Hq above its fixed scratch (2,097,152) */
#define ATTN_ERR_WORKSPACE (-14)     /* workspace below its minimum size (T * Hq floats, 256-byte padded) */
#define ATTN_ERR_STRIDE (-15)        /* *_strided: a stride pair that is not a valid [T, H, 128] view */

/* Device status words (attn_varlen_get_status). */
#define ATTN_STATUS_TIMEOUT 1          /* a bounded wait inside a kernel gave up */
#define ATTN_STATUS_LIST_OVERFLOW 2    /* a CTA's work list did not fit */
#define ATTN_STATUS_SMEM_ALIGN 3       /* dynamic shared memory not 1024-byte aligned (internal error) */
#define ATTN_STATUS_SEGMENT_TOO_LONG 4 /* a segment of cu_seqlens is longer than max_seqlen */
#define ATTN_STATUS_GATE_RANGE 5       /* kda_varlen_*: a log decay g at or below -5.8, or NaN */

/*
 * Forward.  Writes out [T, Hq, 128] (bf16) and lse [Hq, T] (float32).
 * softmax_scale is normally 1/sqrt(128).  max_seqlen is an upper bound on
 * every segment length (the context length is a valid, graph-friendly choice).
 */
int attn_varlen_fwd(const void* q, const void* k, const void* v, const int32_t* cu_seqlens, int32_t max_seqlen,
                    int32_t window_left, float softmax_scale, void* out, float* lse, int64_t total,
                    int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, int32_t num_segments,
                    void* stream);

/*
 * Backward.  Given dout, the forward's inputs and its outputs out and lse,
 * writes dq [T, Hq, 128], dk and dv [T, Hkv, 128] (bf16).  Runs four kernels
 * on `stream`: a preprocess computing D = rowsum(dout * out), a one-CTA
 * planner writing the longest-first work lists (beside the preprocess), a
 * key/value-stationary pass producing dk and dv, and a query-stationary pass
 * producing dq.  No floating-point atomics: results are bitwise reproducible
 * (the passes' CTAs claim work units at run time, but no sum depends on
 * which CTA computes which unit).
 */
int attn_varlen_bwd(const void* dout, const void* q, const void* k, const void* v, const void* out,
                    const float* lse, const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left,
                    float softmax_scale, void* dq, void* dk, void* dv, int64_t total, int32_t num_heads_q,
                    int32_t num_heads_kv, int32_t head_dim, int32_t num_segments, void* stream);

/*
 * The backward for callers that cannot allocate device memory.  (The page
 * has no counterpart; this is a property of the library, not of the method.)
 * Some callers may not call cudaMalloc or the stream-ordered allocator: code
 * running under an allocator it does not own (a framework's caching
 * allocator, a fixed pre-reserved memory budget), real-time or embedded
 * callers for which a driver allocation may block or synchronise the device,
 * or paths that must not allocate at all.  This call runs the same three
 * kernels as attn_varlen_bwd, with the same arguments and launch order, and
 * gives the same bits, but keeps its scratch (D = rowsum(dout * out), float32
 * [Hq, T], and the dK/dV pass's chain buffers) in a fixed device array
 * compiled into the library instead of allocating it; it calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   Limit: T * Hq <= 2,097,152.  The array is 52,693,760 bytes (8 MiB of D,
 *   the counters and work lists of the two passes, and the 320 chain
 *   buffers of 128 KiB that attn_varlen_bwd also uses); larger problems return
 *   ATTN_ERR_NOALLOC_TOO_LARGE before anything is enqueued.  Every GPU that
 *   loads the library holds the array until the process exits.
 *   Sharing: all calls on a device use the same array.  The previous call's
 *   contents are irrelevant (D is overwritten and the chain counters are
 *   reset at the start of every call), but calls whose GPU work overlaps in
 *   time (different streams or host threads) race on the array; the caller
 *   must order them.
 *   Set-up: the first call on each device looks up the array's device
 *   address (with that device current) and caches it; make that first call
 *   before any stream capture.
 */
int attn_varlen_bwd_noalloc(const void* dout, const void* q, const void* k, const void* v, const void* out,
                            const float* lse, const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left,
                            float softmax_scale, void* dq, void* dk, void* dv, int64_t total, int32_t num_heads_q,
                            int32_t num_heads_kv, int32_t head_dim, int32_t num_segments, void* stream);

/*
 * The forward and backward on strided views, so that a layer can hand over
 * its tensors as they come out of its projections and take the gradients
 * straight into its own buffers (research.dws.rip/llm/kernels, section 06 and
 * Fig. 8: one attention layer with its projections and a small loss, replayed
 * as a CUDA graph).  For example q, k and v can be the three head ranges of
 * one fused [T, Hq + 2 Hkv, 128] projection output, and dq, dk, dv the same
 * ranges of its gradient.
 *
 * Same arguments and results as attn_varlen_fwd / attn_varlen_bwd, plus
 * `strides`: host int64 pairs (token stride, head stride) in elements, one
 * pair per [T, H, 128] tensor, in the order
 *     forward:  q, k, v, out                          (8 values)
 *     backward: dout, q, k, v, out, dq, dk, dv        (16 values)
 * Element (t, h, c) of a tensor lives at base + t * token + h * head + c.
 * Each stride is a positive multiple of 8 elements (16 bytes), head >= 128,
 * token >= head * H; otherwise the call returns ATTN_ERR_STRIDE before
 * enqueueing anything.  Output views must not overlap each other or the
 * inputs.  lse stays a dense float32 [Hq, T].  The array is read during the
 * call only.
 */
int attn_varlen_fwd_strided(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                            int32_t max_seqlen, int32_t window_left, float softmax_scale, void* out, float* lse,
                            int64_t total, int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim,
                            int32_t num_segments, const int64_t* strides, void* stream);
int attn_varlen_bwd_strided(const void* dout, const void* q, const void* k, const void* v, const void* out,
                            const float* lse, const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left,
                            float softmax_scale, void* dq, void* dk, void* dv, int64_t total, int32_t num_heads_q,
                            int32_t num_heads_kv, int32_t head_dim, int32_t num_segments, const int64_t* strides,
                            void* stream);

/* Bytes of scratch the backward takes from the stream-ordered allocator:
 * D (T * Hq floats, 256-byte padded), 2,816 bytes of counters, two lists of
 * work items the passes claim at run time (2 x 32,768 x 36 bytes), and 40 MiB
 * of chain buffers.  0 when total <= 0 or num_heads_q <= 0. */
size_t attn_varlen_bwd_workspace_bytes(int64_t total, int32_t num_heads_q);

/* The same size, taking the arguments a caller passes to the calls
 * (num_segments and max_seqlen do not change it; negative values give 0). */
size_t attn_varlen_workspace_bytes(int64_t total, int32_t num_heads_q, int32_t num_segments, int32_t max_seqlen);

/*
 * Registers a caller-owned device buffer as the backward's scratch on the
 * current device (the page's training loop replays a graph over fixed
 * memory: research.dws.rip/llm/kernels, section 06).  From then on
 * attn_varlen_bwd and attn_varlen_bwd_strided on this device use it, with
 * the same kernels, launch order and overlap, and allocate nothing.
 * dev_ptr must be 256-byte aligned; with
 * attn_varlen_bwd_workspace_bytes() bytes the results are the same bits as
 * with the library's own scratch, a smaller buffer (at least T * Hq floats,
 * 256-byte padded, else a call returns ATTN_ERR_WORKSPACE) splits long
 * key/value tiles less.  dev_ptr = NULL or bytes = 0 goes back to the
 * library's own scratch.  The buffer must stay valid while calls that use it
 * run; calls on one device whose GPU work overlaps race on it.  The library
 * does not free it.  Returns ATTN_ERR_ALIGNMENT for a misaligned pointer,
 * ATTN_ERR_DEVICE if the current device is not an sm_103 GPU.
 */
int attn_varlen_set_workspace(void* dev_ptr, size_t bytes);

/*
 * The kernels of attn_varlen_bwd as separate calls, for callers that manage
 * the scratch themselves.  `workspace` is caller-owned device memory, 256-byte
 * aligned, of `workspace_bytes` bytes; the same workspace goes to every call,
 * in this order on one stream:
 *   attn_varlen_bwd_preprocess writes D = rowsum(dout * out) (float32 [Hq, T],
 *     at the start of the workspace) and resets the passes' counters;
 *   attn_varlen_bwd_plan (optional) writes the longest-first work lists of
 *     the two passes into the workspace, from which their CTAs then claim
 *     units at run time; without it every CTA deals itself a fixed share;
 *   attn_varlen_bwd_dkdv reads D (with q, k, v, dout, lse) and writes dk, dv;
 *   attn_varlen_bwd_dq reads D and writes dq.
 * A pass consumes its list: run attn_varlen_bwd_plan again before running it
 * again with lists (without, it falls back to fixed shares, same bits).
 * Minimum size: T * Hq * 4 bytes rounded up to 256.  With
 * attn_varlen_bwd_workspace_bytes() bytes the lists fit and the dK/dV pass
 * may split long key/value tiles into chunks whose partial sums are added in
 * a fixed order (better load balance, same bits); a smaller workspace splits
 * less and claims nothing.  Arguments otherwise mean what they mean in
 * attn_varlen_bwd.
 */
int attn_varlen_bwd_preprocess(const void* dout, const void* out, void* workspace, size_t workspace_bytes,
                               int64_t total, int32_t num_heads_q, int32_t head_dim, void* stream);
int attn_varlen_bwd_plan(const int32_t* cu_seqlens, int32_t max_seqlen, int32_t window_left, void* workspace,
                         size_t workspace_bytes, int64_t total, int32_t num_heads_q, int32_t num_heads_kv,
                         int32_t num_segments, void* stream);
int attn_varlen_bwd_dkdv(const void* dout, const void* q, const void* k, const void* v, const float* lse,
                         const void* workspace, size_t workspace_bytes, const int32_t* cu_seqlens, int32_t max_seqlen,
                         int32_t window_left, float softmax_scale, void* dk, void* dv, int64_t total,
                         int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, int32_t num_segments,
                         void* stream);
int attn_varlen_bwd_dq(const void* dout, const void* q, const void* k, const void* v, const float* lse,
                       const void* workspace, size_t workspace_bytes, const int32_t* cu_seqlens, int32_t max_seqlen,
                       int32_t window_left, float softmax_scale, void* dq, int64_t total, int32_t num_heads_q,
                       int32_t num_heads_kv, int32_t head_dim, int32_t num_segments, void* stream);

/*
 * Synchronises `stream`, then returns ATTN_OK if no kernel of this library
 * recorded an error on the current device since the last call, else
 * ATTN_ERR_DEVICE_STATUS; *device_code (optional) receives the raw word,
 * one of the ATTN_STATUS_* values (the last error recorded).
 * The word is cleared.  For tests and debugging; it blocks the host.
 */
int attn_varlen_get_status(void* stream, int32_t* device_code);

/* Static description of an error code. */
const char* attn_varlen_strerror(int code);

/*
 * Test hook: runs the kernels' own mask and tile-range logic on the device.
 * by_key = 0: for every query token i, ranges[3*i + 0..2] = (first visible
 *   key, last visible key, number of visible keys), scanning exactly the kv
 *   tiles and per-row column bounds the forward and dQ kernels use.
 * by_key = 1: for every key token j, (first query that sees j, last query
 *   that sees j, number of such queries), scanning the q tiles and bounds the
 *   dK/dV kernel uses.
 * A token that sees (or is seen by) nothing gets (0, -1, 0).
 * ranges is device int32 [3 * T].
 */
int attn_varlen_mask_ranges(const int32_t* cu_seqlens, int32_t num_segments, int64_t total, int32_t max_seqlen,
                            int32_t window_left, int32_t by_key, int32_t* ranges, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_VARLEN_H_ */
