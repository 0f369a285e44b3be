/*
 * gdn_varlen.h -- C ABI of the Gated DeltaNet local layer over packed
 * documents, in the same GB300 (sm_103a) library as attn_varlen.h
 * (libvsw_attn.so; error codes and the device status word are shared).
 *
 * The operation.  research.dws.rip/llm/kernels, section 03 "What linear
 * attention costs", weighs Gated DeltaNet (Yang et al., "Gated Delta
 * Networks: Improving Mamba2 with Delta Rule") against the sliding window as
 * the local layer, on the same 16,384-token microbatches packed from
 * documents (section 01).  The pages give no formula; this is the published
 * recurrence, per head, with the state kept as a d_k x d_v matrix H:
 *     alpha_t = exp(g_t)
 *     e_t     = beta_t (v_t - alpha_t H_{t-1}^T k_t)
 *     H_t     = alpha_t H_{t-1} + k_t e_t^T
 *     o_t     = scale * H_t^T q_t
 * with H = 0 at the first token of every segment [cu_seqlens[s],
 * cu_seqlens[s+1]) (no state crosses a document boundary or row cut; empty
 * segments change no output bit).  q and k are taken as given: the layer
 * around the kernel L2-normalises them.
 *
 * Layouts (row-major, contiguous):
 *     q, k, v, o : bf16 [T, H, 128]        g, beta : float32 [T, H]
 *     cu_seqlens : int32 [num_segments + 1], as in attn_varlen.h
 * g is the log of the decay (<= 0 in a layer; any finite value is computed
 * as given), beta the write strength.
 *
 * Method: chunks of 64 tokens aligned to each segment's start.  Per chunk
 * and head the WY form of the 64 delta-rule steps (a unit lower-triangular
 * 64 x 64 inverse) is built in parallel; then one pass per (segment, head,
 * 32 value columns) carries the state across the segment's chunks and writes
 * o.  The backward recomputes that, carries the state's gradient back across
 * the chunks the same way, and then forms every chunk's gradients in
 * parallel.  Matrix products run on tensor cores in bf16 with float32
 * accumulation; states and their gradients stay float32 along the chains.
 *
 * Ownership: every pointer is caller-owned device memory on the current
 * device, 16-byte aligned (workspace: 256-byte aligned), and `stream` is a
 * cudaStream_t passed as void*.  Nothing is allocated and the host is never
 * synchronised; the call is CUDA-graph capturable.  Returns ATTN_OK or a
 * negative ATTN_ERR_* code (attn_varlen.h) before anything is enqueued.
 */
#ifndef GDN_VARLEN_H_
#define GDN_VARLEN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of device workspace gdn_varlen_fwd needs for T tokens, H heads and
 * num_segments segments: the chunk and segment tables, the per-chunk WY
 * factors W and U (bf16 [T, H, 128] each), the masked intra-chunk q.k
 * products (bf16 64 x 64 per chunk and head) and the running log decay
 * (float32 [H, T]).  0 for invalid sizes. */
size_t gdn_varlen_workspace_bytes(int64_t total, int32_t num_heads, int32_t num_segments);

/* o = the recurrence above, for all heads and segments.
 * q, k, v: bf16 [T, H, head_dim]; g, beta: float32 [T, H]; o: bf16
 * [T, H, head_dim], fully overwritten.  scale: finite (1/sqrt(128) in a
 * layer).  workspace: at least gdn_varlen_workspace_bytes(T, H, num_segments)
 * bytes, contents need not be initialised, used only by the enqueued work.
 * Errors: ATTN_ERR_NULL_POINTER, ATTN_ERR_SHAPE (T < 0, H <= 0,
 * num_segments < 0, or num_segments = 0 with T > 0), ATTN_ERR_HEAD_DIM
 * (head_dim != 128), ATTN_ERR_ALIGNMENT, ATTN_ERR_SCALE (not finite),
 * ATTN_ERR_TOO_LARGE, ATTN_ERR_WORKSPACE (too small), ATTN_ERR_DEVICE,
 * ATTN_ERR_CUDA. */
int gdn_varlen_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                   const int32_t* cu_seqlens, float scale, void* o, void* workspace, size_t workspace_bytes,
                   int64_t total, int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream);

/* Bytes of device workspace gdn_varlen_bwd needs: the forward's, plus the
 * bf16 state at every chunk start and its gradient at every chunk end
 * ([chunks, H, 128, 128] each, chunks <= T / 64 + num_segments + 1), the
 * chunks' pseudo-values E and the gradients dE, dW (bf16 [T, H, 128] each),
 * a float32 [T, H, 128] part of dk and a float32 [H, T] part of dg.
 * 0 for invalid sizes. */
size_t gdn_varlen_bwd_workspace_bytes(int64_t total, int32_t num_heads, int32_t num_segments);

/* Gradients of L = sum(d_o * o) for the forward above: dq, dk, dv (bf16
 * [T, H, 128]) and dg, dbeta (float32 [T, H]), all fully overwritten.  d_o:
 * bf16 [T, H, 128].  The forward is recomputed inside (o itself is not
 * needed).  workspace: at least gdn_varlen_bwd_workspace_bytes(T, H,
 * num_segments) bytes, 256-byte aligned.  Same error codes as
 * gdn_varlen_fwd. */
int gdn_varlen_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta, const void* d_o,
                   const int32_t* cu_seqlens, float scale, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                   void* workspace, size_t workspace_bytes, int64_t total, int32_t num_heads, int32_t head_dim,
                   int32_t num_segments, void* stream);

/* A training step's pair: the forward above that also keeps, in a workspace
 * sized for the backward, everything the backward would recompute (the
 * chunk tables, the WY factors, the state at every chunk start and every
 * chunk's E), and the backward that reads them instead.  Same results, bit
 * for bit, as gdn_varlen_fwd and gdn_varlen_bwd; the backward saves the plan,
 * the prep pass and the recomputing state pass.
 *
 * gdn_varlen_fwd_save: the arguments of gdn_varlen_fwd, with workspace of at
 * least gdn_varlen_bwd_workspace_bytes(T, H, num_segments) bytes.
 * gdn_varlen_bwd_saved: the arguments of gdn_varlen_bwd.  It trusts the
 * workspace: it must be the one the last gdn_varlen_fwd_save on this stream
 * wrote, with the same q, k, v, g, beta, cu_seqlens, scale and sizes, and no
 * other call may have used it in between.  Otherwise the gradients are
 * meaningless, though every access stays inside the caller's buffers.
 * Error codes as the calls they pair. */
int gdn_varlen_fwd_save(const void* q, const void* k, const void* v, const float* g, const float* beta,
                        const int32_t* cu_seqlens, float scale, void* o, void* workspace, size_t workspace_bytes,
                        int64_t total, int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream);
int gdn_varlen_bwd_saved(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const void* d_o, const int32_t* cu_seqlens, float scale, void* dq, void* dk, void* dv,
                         float* dg, float* dbeta, void* workspace, size_t workspace_bytes, int64_t total,
                         int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_VARLEN_H_ */
