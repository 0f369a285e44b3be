/*
 * kda_varlen.h -- C ABI of the Kimi Delta attention local layer over packed
 * documents, in the same GB300 (sm_103a) library as attn_varlen.h and
 * gdn_varlen.h (libvsw_attn.so; error codes and the device status word are
 * shared).
 *
 * The operation.  research.dws.rip/llm/kernels, section 03 "What linear
 * attention costs", weighs Kimi Delta attention (the Kimi Linear model's
 * local layer) against the sliding window on the same packed microbatches;
 * the pages record it as the layer that was kept.  They give no formula; this
 * is the published one, the gated delta rule with a decay per key channel,
 * per head, with the state S of d_k x d_v:
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t,            alpha_t = exp(g_t), g_t in R^{d_k}
 * with S = 0 at the first token of every segment [cu_seqlens[s],
 * cu_seqlens[s+1]) (empty segments change no output bit).  q and k are taken
 * as given: the layer around the kernel L2-normalises them.  With every
 * channel of g equal it is the Gated DeltaNet of gdn_varlen.h.
 *
 * Layouts (row-major, contiguous):
 *     q, k, v, o : bf16 [T, H, 128]     g : float32 [T, H, 128]    beta : float32 [T, H]
 *     cu_seqlens : int32 [num_segments + 1], as in attn_varlen.h
 * g is the log decay per token, head and key channel.  The kernels split each
 * chunk's decay at the start of every 16-token block, so the decay over 15
 * tokens of one channel must stay inside float range: every g > -5.8 (a
 * per-token decay above 0.003).  The kernels check this: a chunk holding a g
 * at or below -5.8 (or a NaN) sets the device status word to
 * ATTN_STATUS_GATE_RANGE (attn_varlen_get_status), and its outputs are then
 * not to be trusted.
 *
 * Method: as gdn_varlen.h, chunks of 64 tokens and the WY form of the
 * chunk's delta-rule steps, with the decay applied per channel inside the
 * products.  Ownership, streams and errors: as gdn_varlen.h.
 */
#ifndef KDA_VARLEN_H_
#define KDA_VARLEN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of device workspace kda_varlen_fwd needs for T tokens, H heads and
 * num_segments segments: the Gated DeltaNet forward's, plus Q o e^gamma and
 * K o e^(gamma_last - gamma) (bf16 [T, H, 128] each) and every chunk's total
 * decay per channel (float32 [chunks, H, 128]).  0 for invalid sizes. */
size_t kda_varlen_workspace_bytes(int64_t total, int32_t num_heads, int32_t num_segments);

/* o = the recurrence above.  q, k, v: bf16 [T, H, head_dim]; g: float32
 * [T, H, head_dim]; beta: float32 [T, H]; o: bf16 [T, H, head_dim], fully
 * overwritten.  Error codes as gdn_varlen_fwd. */
int kda_varlen_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                   const int32_t* cu_seqlens, float scale, void* o, void* workspace, size_t workspace_bytes,
                   int64_t total, int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream);

/* Bytes of device workspace kda_varlen_bwd needs: the forward's and the
 * Gated DeltaNet backward's, plus per chunk and head X = (I + A)^-1, the
 * unscaled A, and the gradients of the masked q.k block and of A (float32
 * 64 x 64 each), and float32 [T, H, 128] parts of dq and of dg.  0 for
 * invalid sizes. */
size_t kda_varlen_bwd_workspace_bytes(int64_t total, int32_t num_heads, int32_t num_segments);

/* Gradients of L = sum(d_o * o): dq, dk, dv (bf16 [T, H, 128]), dg (float32
 * [T, H, 128], one per key channel) and dbeta (float32 [T, H]), all fully
 * overwritten; the forward is recomputed inside.  Error codes as
 * gdn_varlen_bwd. */
int kda_varlen_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta, const void* d_o,
                   const int32_t* cu_seqlens, float scale, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                   void* workspace, size_t workspace_bytes, int64_t total, int32_t num_heads, int32_t head_dim,
                   int32_t num_segments, void* stream);

/* The training step's pair, as gdn_varlen_fwd_save / gdn_varlen_bwd_saved:
 * kda_varlen_fwd_save takes the arguments of kda_varlen_fwd with a workspace
 * of at least kda_varlen_bwd_workspace_bytes(T, H, num_segments) bytes and
 * also keeps X, the unscaled A, the states and E there; kda_varlen_bwd_saved
 * takes the arguments of kda_varlen_bwd and trusts that workspace the same
 * way.  Same results, bit for bit, as kda_varlen_fwd and kda_varlen_bwd. */
int kda_varlen_fwd_save(const void* q, const void* k, const void* v, const float* g, const float* beta,
                        const int32_t* cu_seqlens, float scale, void* o, void* workspace, size_t workspace_bytes,
                        int64_t total, int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream);
int kda_varlen_bwd_saved(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const void* d_o, const int32_t* cu_seqlens, float scale, void* dq, void* dk, void* dv,
                         float* dg, float* dbeta, void* workspace, size_t workspace_bytes, int64_t total,
                         int32_t num_heads, int32_t head_dim, int32_t num_segments, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_VARLEN_H_ */
