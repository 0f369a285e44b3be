"""Plain float64 CPU oracle for the Gated DeltaNet recurrence over packed
documents (the linear-attention local layer the pages weigh against the
sliding window).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this module.  The library's product
path never calls it, and it shares no code with the CUDA kernels.

What it computes.  research.dws.rip/llm/kernels, section 03 "What linear
attention costs", pits Gated DeltaNet (Yang et al., "Gated Delta Networks:
Improving Mamba2 with Delta Rule") against the window on the same packed
16,384-token microbatches, checked against a token-by-token reference; section
06 (Fig. 8) replays it with boundary lists padded by empty documents.  The
pages give no formula, so the recurrence is the published one, with the state
kept as a d_k x d_v matrix H (the transpose of the paper's S):

    alpha_t = exp(g_t)                          (g_t <= 0, one gate per token and head)
    e_t     = beta_t (v_t - alpha_t H_{t-1}^T k_t)
    H_t     = alpha_t H_{t-1} + k_t e_t^T       (= alpha_t (I - beta_t k_t k_t^T) H_{t-1} + beta_t k_t v_t^T)
    o_t     = scale * H_t^T q_t

per head, with H = 0 at the first token of every segment (document
masking: no state crosses a boundary; empty segments do nothing).

Readings where the pages are silent (each also listed in the design notes):
  * q and k arrive already L2-normalised (the layer normalises them before the
    kernel); the kernel takes them as given.  scale = 1/sqrt(d_k) by default.
  * g is the log of the decay (fp32, <= 0) and beta the write strength (fp32,
    in (0, 1)), both [T, H].
  * heads: H heads of d_k = d_v = 128, no grouping (the same 8 x 128 as the
    attention layer's query heads).

The backward is reverse-mode differentiation of exactly these steps, token by
token, for L = sum <do, o>.  States are kept at every CHECKPOINT-th token and
recomputed in between, to bound memory on long segments.

Pins (tests/test_oracle_gdn.py): central finite differences of every input,
closed forms (alpha = 0, beta = 0, orthogonal keys = causal linear attention,
one repeated unit key = last-write-wins memory), segment isolation, empty
segments, a chunked (WY-form) evaluation written independently in the test,
and torch float64 autograd through the same recurrence.
"""
from __future__ import annotations

import numpy as np

CHECKPOINT = 64


def segments(cu_seqlens):
    """Yields (a, b) for every non-empty segment."""
    cu = [int(x) for x in cu_seqlens]
    for a, b in zip(cu[:-1], cu[1:]):
        if b > a:
            yield a, b


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _step(Hs, q, k, v, g, beta, scale):
    """One token for all heads.  Hs [H, dk, dv] is updated in place; returns o [H, dv]."""
    alpha = np.exp(g)                                   # [H]
    pred = alpha[:, None] * np.einsum("hkv,hk->hv", Hs, k)
    e = beta[:, None] * (v - pred)
    Hs *= alpha[:, None, None]
    Hs += k[:, :, None] * e[:, None, :]
    return scale * np.einsum("hkv,hk->hv", Hs, q)


def forward(q, k, v, g, beta, cu_seqlens, scale=None, return_states=False):
    """o [T, H, dv] (float64) of the recurrence above; with return_states, also
    the final state [H, dk, dv] of every non-empty segment, in order."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    T, nh, dk = k.shape
    dv = v.shape[2]
    scale = 1.0 / np.sqrt(dk) if scale is None else float(scale)
    o = np.zeros((T, nh, dv))
    finals = []
    for a, b in segments(cu_seqlens):
        Hs = np.zeros((nh, dk, dv))
        for t in range(a, b):
            o[t] = _step(Hs, q[t], k[t], v[t], g[t], beta[t], scale)
        finals.append(Hs.copy())
    return (o, finals) if return_states else o


def backward(q, k, v, g, beta, do, cu_seqlens, scale=None):
    """Gradients (dq, dk, dv, dg, dbeta) of L = sum <do, o>, float64."""
    q, k, v, g, beta, do = (_f64(x) for x in (q, k, v, g, beta, do))
    T, nh, dk = k.shape
    dv_ = v.shape[2]
    scale = 1.0 / np.sqrt(dk) if scale is None else float(scale)
    dq, dk_, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dg, dbeta = np.zeros_like(g), np.zeros_like(beta)
    for a, b in segments(cu_seqlens):
        # Forward once, keeping the state before every CHECKPOINT-th token.
        starts = list(range(a, b, CHECKPOINT))
        ck = {}
        Hs = np.zeros((nh, dk, dv_))
        for t in range(a, b):
            if (t - a) % CHECKPOINT == 0:
                ck[t] = Hs.copy()
            _step(Hs, q[t], k[t], v[t], g[t], beta[t], scale)
        dH = np.zeros((nh, dk, dv_))  # gradient w.r.t. H_t from the tokens after t
        for s0 in reversed(starts):
            s1 = min(b, s0 + CHECKPOINT)
            # States H_{t-1} for t in [s0, s1), recomputed from the checkpoint.
            prev = []
            Hs = ck[s0].copy()
            for t in range(s0, s1):
                prev.append(Hs.copy())
                _step(Hs, q[t], k[t], v[t], g[t], beta[t], scale)
            Ht = Hs  # H_{s1 - 1}
            for t in range(s1 - 1, s0 - 1, -1):
                Hp = prev[t - s0]
                alpha, bt = np.exp(g[t]), beta[t]
                Hk = np.einsum("hkv,hk->hv", Hp, k[t])          # H_{t-1}^T k_t
                pred = alpha[:, None] * Hk
                r = v[t] - pred
                e = bt[:, None] * r
                # o_t = scale H_t^T q_t
                dq[t] = scale * np.einsum("hkv,hv->hk", Ht, do[t])
                dH += scale * q[t][:, :, None] * do[t][:, None, :]
                # H_t = alpha H_{t-1} + k e^T
                de = np.einsum("hkv,hk->hv", dH, k[t])
                dk_[t] += np.einsum("hkv,hv->hk", dH, e)
                dalpha = np.einsum("hkv,hkv->h", dH, Hp)
                dHp = alpha[:, None, None] * dH
                # e = beta (v - alpha H_{t-1}^T k)
                dbeta[t] = np.einsum("hv,hv->h", de, r)
                dv[t] = bt[:, None] * de
                dpred = -bt[:, None] * de
                dalpha += np.einsum("hv,hv->h", dpred, Hk)
                dHp += alpha[:, None, None] * k[t][:, :, None] * dpred[:, None, :]
                dk_[t] += alpha[:, None] * np.einsum("hkv,hv->hk", Hp, dpred)
                dg[t] = dalpha * alpha
                dH = dHp
                Ht = Hp
    return dq, dk_, dv, dg, dbeta
