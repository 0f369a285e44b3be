"""Plain float64 CPU oracle for Kimi Delta attention over packed documents
(the local layer that won the pages' bake-off).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this module.  The library's product
path never calls it, and it shares no code with the CUDA kernels.

What it computes.  research.dws.rip/llm/kernels, section 03 "What linear
attention costs", weighs Kimi Delta Attention (the Kimi Linear model's local
layer) against the window on the same packed microbatches, checked against a
token-by-token reference; the last table of the pages records it as the
layer that was kept.  The pages give no formula; this is the published one:
the gated delta rule with a decay per key channel,

    S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = scale * S_t^T q_t,          alpha_t = exp(g_t) in R^{d_k}

(S of d_k x d_v), written here as the equivalent update

    e_t = beta_t (v_t - S_{t-1}^T (alpha_t o k_t)),
    S_t = Diag(alpha_t) S_{t-1} + k_t e_t^T,

per head, with S = 0 at the first token of every segment.

Readings (also in the design notes): q and k arrive L2-normalised; g is the
log decay per token, head and key channel, float32 [T, H, d_k]; beta float32
[T, H]; with every channel of g equal it is Gated DeltaNet (gated_delta.py).

The backward is reverse-mode differentiation of these steps, token by token,
for L = sum <do, o>, with states checkpointed every CHECKPOINT tokens.

Pins (tests/test_oracle_kda.py): central finite differences of every input,
torch float64 autograd through the paper's form of the step, equality with
the Gated DeltaNet oracle when the gate is the same on every channel, closed
forms, segment isolation, empty segments, and a chunked evaluation written
in the test from the algebra.
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


def _step(S, q, k, v, g, beta, scale):
    """One token for all heads.  S [H, dk, dv] is updated in place; returns o [H, dv]."""
    alpha = np.exp(g)                                    # [H, dk]
    pred = np.einsum("hkv,hk->hv", S, alpha * k)         # S^T (alpha o k)
    e = beta[:, None] * (v - pred)
    S *= alpha[:, :, None]
    S += k[:, :, None] * e[:, None, :]
    return scale * np.einsum("hkv,hk->hv", S, q)


def forward(q, k, v, g, beta, cu_seqlens, scale=None):
    """o [T, H, dv] (float64)."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    T, nh, dk = k.shape
    dv = v.shape[2]
    scale = 1.0 / np.sqrt(dk) if scale is None else float(scale)
    o = np.zeros((T, nh, dv))
    for a, b in segments(cu_seqlens):
        S = np.zeros((nh, dk, dv))
        for t in range(a, b):
            o[t] = _step(S, q[t], k[t], v[t], g[t], beta[t], scale)
    return o


def backward(q, k, v, g, beta, do, cu_seqlens, scale=None):
    """Gradients (dq, dk, dv, dg, dbeta) of L = sum <do, o>, float64; dg has
    the shape of g ([T, H, dk])."""
    q, k, v, g, beta, do = (_f64(x) for x in (q, k, v, g, beta, do))
    T, nh, dk = k.shape
    dv_ = v.shape[2]
    scale = 1.0 / np.sqrt(dk) if scale is None else float(scale)
    dq, dk_, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dg, dbeta = np.zeros_like(g), np.zeros_like(beta)
    for a, b in segments(cu_seqlens):
        starts = list(range(a, b, CHECKPOINT))
        ck = {}
        S = np.zeros((nh, dk, dv_))
        for t in range(a, b):
            if (t - a) % CHECKPOINT == 0:
                ck[t] = S.copy()
            _step(S, q[t], k[t], v[t], g[t], beta[t], scale)
        dS = np.zeros((nh, dk, dv_))  # gradient w.r.t. S_t from the tokens after t
        for s0 in reversed(starts):
            s1 = min(b, s0 + CHECKPOINT)
            prev = []
            S = ck[s0].copy()
            for t in range(s0, s1):
                prev.append(S.copy())
                _step(S, q[t], k[t], v[t], g[t], beta[t], scale)
            St = S
            for t in range(s1 - 1, s0 - 1, -1):
                Sp = prev[t - s0]
                alpha, bt = np.exp(g[t]), beta[t]
                ak = alpha * k[t]
                pred = np.einsum("hkv,hk->hv", Sp, ak)
                r = v[t] - pred
                e = bt[:, None] * r
                # o_t = scale S_t^T q_t
                dq[t] = scale * np.einsum("hkv,hv->hk", St, do[t])
                dS += scale * q[t][:, :, None] * do[t][:, None, :]
                # S_t = Diag(alpha) S_{t-1} + k e^T
                de = np.einsum("hkv,hk->hv", dS, k[t])
                dk_[t] += np.einsum("hkv,hv->hk", dS, e)
                dalpha = np.einsum("hkv,hkv->hk", dS, Sp)
                dSp = alpha[:, :, None] * dS
                # e = beta (v - S_{t-1}^T (alpha o k))
                dbeta[t] = np.einsum("hv,hv->h", de, r)
                dv[t] = bt[:, None] * de
                dpred = -bt[:, None] * de
                dak = np.einsum("hkv,hv->hk", Sp, dpred)
                dSp += ak[:, :, None] * dpred[:, None, :]
                dalpha += dak * k[t]
                dk_[t] += dak * alpha
                dg[t] = dalpha * alpha
                dS = dSp
                St = Sp
    return dq, dk_, dv, dg, dbeta
