"""Plain float64 CPU oracle for document-masked causal grouped-query attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this module.  The library's product
path never calls it, and it shares no code with the CUDA kernels.

What it computes, read from research.dws.rip/llm/kernels:
  * section 01 "How it was measured": a microbatch is packed from documents,
    no document attends across its own boundary and every row is cut at the
    context length, so attention is restricted to segments;
  * Fig. 2 "Benchmark setup": 8 query heads and 2 key-value heads of width 128
    (grouped-query attention), and a 512-token window on the local layers;
  * section 01 again: outputs *and gradients* are checked against a
    higher-precision reference, so the oracle gives the forward and the
    analytic backward.

Readings where the page is silent (each also listed in the design notes):
  * window_left = w >= 0 means key j is visible from query i iff
    i - w <= j <= i (w+1 keys including the query itself); w = -1 is
    global causal.  The window never reaches across a segment boundary.
  * query head h reads key/value head h // (Hq // Hkv).
  * lse is the natural log-sum-exp of the scaled logits, [Hq, T].
  * empty segments (repeated boundaries) contribute nothing.

Definition, per segment [a, b), head h, kv head g, query i in [a, b):
    V(i)      = { j : a <= j <= i and (w < 0 or i - j <= w) }
    s_ij      = scale * <q[i,h], k[j,g]>
    lse_i     = log sum_{j in V(i)} exp(s_ij)
    P_ij      = exp(s_ij - lse_i)
    out[i,h]  = sum_{j in V(i)} P_ij v[j,g]
and the backward of L = sum <dout, out>:
    dP_ij = <dout[i,h], v[j,g]>,  D_i = sum_j P_ij dP_ij,
    dS_ij = P_ij (dP_ij - D_i)
    dq[i,h] = scale sum_j dS_ij k[j,g]
    dk[j,g] = scale sum_{h in group g} sum_i dS_ij q[i,h]
    dv[j,g] =       sum_{h in group g} sum_i P_ij dout[i,h]

Every function below is written straight from these formulas with an explicit
boolean mask per segment; long segments are cut into blocks of query rows only
to bound memory.  Pins (tests/test_oracle.py): finite differences, closed
forms, invariants, hand-derived fixtures and torch's float64 SDPA.
"""
from __future__ import annotations

import numpy as np

ROW_BLOCK = 1024


def segments(cu_seqlens):
    """Yields (a, b) for every non-empty segment."""
    cu = [int(x) for x in cu_seqlens]
    for a, b in zip(cu[:-1], cu[1:]):
        if b > a:
            yield a, b


def visible_mask(a: int, b: int, window_left: int, r0: int | None = None, r1: int | None = None) -> np.ndarray:
    """Boolean [rows, b-a]: entry (i, j) is True iff key a+j is in V(i).

    Rows are the queries a+r0 .. a+r1-1 of the segment [a, b).
    """
    L = b - a
    r0 = 0 if r0 is None else r0
    r1 = L if r1 is None else r1
    i = np.arange(r0, r1)[:, None]
    j = np.arange(L)[None, :]
    m = j <= i
    if window_left >= 0:
        m &= (i - j) <= window_left
    return m


def visible_ranges(cu_seqlens, window_left: int, total: int) -> np.ndarray:
    """For every token i: (first visible key, last visible key, |V(i)|), int64 [T, 3].

    Tokens outside every segment (none, for a valid cu_seqlens) get (0, -1, 0).
    """
    out = np.zeros((total, 3), dtype=np.int64)
    out[:, 1] = -1
    for a, b in segments(cu_seqlens):
        for r in range(b - a):
            row = visible_mask(a, b, window_left, r, r + 1)[0]
            idx = np.nonzero(row)[0]
            out[a + r] = (a + idx[0], a + idx[-1], idx.size)
    return out


def _group(hq: int, hkv: int, h: int) -> int:
    return h // (hq // hkv)


def _segment_head_probs(qs: np.ndarray, ks: np.ndarray, mask: np.ndarray, scale: float):
    """P and lse for one block of query rows of one segment and head."""
    s = scale * (qs @ ks.T)
    s = np.where(mask, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
    p = np.exp(s - lse[:, None])
    return p, lse


def probabilities(q, k, cu_seqlens, window_left: int, softmax_scale: float, seg_index: int, h: int) -> np.ndarray:
    """The full P matrix [L, L] of one (non-empty) segment and query head."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    hq, hkv = q.shape[1], k.shape[1]
    a, b = list(segments(cu_seqlens))[seg_index]
    g = _group(hq, hkv, h)
    p, _ = _segment_head_probs(q[a:b, h], k[a:b, g], visible_mask(a, b, window_left), softmax_scale)
    return p


def forward(q, k, v, cu_seqlens, window_left: int, softmax_scale: float):
    """Returns (out [T, Hq, d], lse [Hq, T]) in float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, hq, d = q.shape
    hkv = k.shape[1]
    out = np.zeros((T, hq, d))
    lse = np.full((hq, T), -np.inf)
    for a, b in segments(cu_seqlens):
        L = b - a
        for r0 in range(0, L, ROW_BLOCK):
            r1 = min(L, r0 + ROW_BLOCK)
            mask = visible_mask(a, b, window_left, r0, r1)
            kcols = r1  # keys after the last row of the block are never visible
            for h in range(hq):
                g = _group(hq, hkv, h)
                p, l = _segment_head_probs(q[a + r0:a + r1, h], k[a:a + kcols, g], mask[:, :kcols], softmax_scale)
                out[a + r0:a + r1, h] = p @ v[a:a + kcols, g]
                lse[h, a + r0:a + r1] = l
    return out, lse


def backward(dout, q, k, v, cu_seqlens, window_left: int, softmax_scale: float):
    """Returns (dq, dk, dv) in float64 for L = sum(dout * out)."""
    dout = np.asarray(dout, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, hq, d = q.shape
    hkv = k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for a, b in segments(cu_seqlens):
        L = b - a
        for r0 in range(0, L, ROW_BLOCK):
            r1 = min(L, r0 + ROW_BLOCK)
            mask = visible_mask(a, b, window_left, r0, r1)
            kc = r1
            for h in range(hq):
                g = _group(hq, hkv, h)
                qi = q[a + r0:a + r1, h]
                doi = dout[a + r0:a + r1, h]
                kj = k[a:a + kc, g]
                vj = v[a:a + kc, g]
                p, _ = _segment_head_probs(qi, kj, mask[:, :kc], softmax_scale)
                dp = doi @ vj.T
                D = (p * dp).sum(axis=1)
                ds = p * (dp - D[:, None])
                dq[a + r0:a + r1, h] = softmax_scale * (ds @ kj)
                dk[a:a + kc, g] += softmax_scale * (ds.T @ qi)
                dv[a:a + kc, g] += p.T @ doi
    return dq, dk, dv


def unmasked_pairs(cu_seqlens, window_left: int) -> int:
    """sum over queries of |V(i)|, by enumerating each segment's mask rows."""
    n = 0
    for a, b in segments(cu_seqlens):
        L = b - a
        for r0 in range(0, L, ROW_BLOCK):
            n += int(visible_mask(a, b, window_left, r0, min(L, r0 + ROW_BLOCK)).sum())
    return n
