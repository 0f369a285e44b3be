"""One attention layer around the library's kernels, with no copies between
them: the fused QKV projection output is handed to the attention as three
strided views, and the attention's gradients land straight in the fused
gradient buffer of that projection (research.dws.rip/llm/kernels, section
06 and Fig. 8: one attention layer plus a small loss, forward and backward,
replayed as a CUDA graph).

    qkv  = x @ W_qkv                   [T, (Hq + 2 Hkv) * 128]
    out  = attention(q, k, v)          q, k, v: head ranges of qkv (views)
    y    = out @ W_o                   [T, D]
    loss = sum(y * g)                  g: a fixed [T, D] weight (the small loss)

and the backward of all of it: dy = g, d_out = dy @ W_o^T, the attention
backward into d_qkv (views again), dW_qkv = x^T @ d_qkv, dW_o = out^T @ dy,
dx = d_qkv @ W_qkv^T.  The projections are plain bf16 GEMMs (torch.matmul,
i.e. cuBLAS); the attention is the library's fwd and bwd through the C ABI.
Every buffer is allocated once, so a step has fixed addresses and shapes and
can be captured in a CUDA graph (with cu_seqlens padded to a fixed count).
"""
from __future__ import annotations

from . import binding


class AttentionLayer:
    """Buffers and weights of one layer for microbatches of `total` tokens."""

    def __init__(self, total: int, d_model: int, hq: int, hkv: int, max_seqlen: int, window_left: int,
                 num_segments: int, seed: int = 0, device="cuda"):
        import torch
        self.total, self.d_model, self.hq, self.hkv = total, d_model, hq, hkv
        self.max_seqlen, self.window_left = max_seqlen, window_left
        self.scale = 128 ** -0.5
        h = hq + 2 * hkv
        gen = torch.Generator(device="cpu").manual_seed(seed)
        bf = torch.bfloat16

        def param(rows, cols):
            w = torch.randn(rows, cols, generator=gen, dtype=torch.float32) / rows ** 0.5
            return w.to(device=device, dtype=bf)
        self.w_qkv = param(d_model, h * 128)
        self.w_o = param(hq * 128, d_model)
        e = lambda *shape, dtype=bf: torch.empty(*shape, dtype=dtype, device=device)  # noqa: E731
        self.x, self.g = e(total, d_model), e(total, d_model)
        self.cu = torch.zeros(num_segments + 1, dtype=torch.int32, device=device)
        self.qkv, self.d_qkv = e(total, h, 128), e(total, h, 128)
        self.out, self.d_out = e(total, hq, 128), e(total, hq, 128)
        self.lse = e(hq, total, dtype=torch.float32)
        self.y = e(total, d_model)
        self.loss = e((), dtype=torch.float32)
        self.dw_qkv, self.dw_o, self.dx = e(*self.w_qkv.shape), e(*self.w_o.shape), e(total, d_model)

    def views(self, t):
        """q, k, v head ranges of a fused [T, Hq + 2 Hkv, 128] buffer."""
        hq, hkv = self.hq, self.hkv
        return t[:, :hq], t[:, hq:hq + hkv], t[:, hq + hkv:]

    def step(self) -> None:
        """Forward and backward of the layer on the current x, g, cu (all on
        the current stream, no host synchronisation)."""
        import torch
        T = self.total
        torch.matmul(self.x, self.w_qkv, out=self.qkv.view(T, -1))
        q, k, v = self.views(self.qkv)
        binding.attn_varlen_fwd(q, k, v, self.cu, self.max_seqlen, self.window_left, self.scale, self.out, self.lse)
        torch.matmul(self.out.view(T, -1), self.w_o, out=self.y)
        self.loss.copy_((self.y.float() * self.g.float()).sum())
        # Backward: dy = g.
        torch.matmul(self.g, self.w_o.t(), out=self.d_out.view(T, -1))
        torch.matmul(self.out.view(T, -1).t(), self.g, out=self.dw_o)
        dq, dk, dv = self.views(self.d_qkv)
        binding.attn_varlen_bwd(self.d_out, q, k, v, self.out, self.lse, self.cu, self.max_seqlen, self.window_left,
                                self.scale, dq, dk, dv)
        torch.matmul(self.x.t(), self.d_qkv.view(T, -1), out=self.dw_qkv)
        torch.matmul(self.d_qkv.view(T, -1), self.w_qkv.t(), out=self.dx)
