"""Shared helpers for the GPU tests: move seeded inputs to the device, run the
library through its C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np

# Relative-L2 tolerances (out and gradients) and the lse bound.
TOL_OUT = 5e-3
TOL_GRAD = 1e-2
TOL_LSE_ABS = 1e-3


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(got.astype(np.float64) - ref) / max(np.linalg.norm(ref), 1e-300))


def segment_errors(got: np.ndarray, ref: np.ndarray, cu_seqlens) -> list[tuple[int, int, float, float]]:
    """Per non-empty segment [a, b) of a token-major tensor: (a, b, ||got - ref||, ||ref||)."""
    got = got.astype(np.float64)
    out = []
    cu = [int(x) for x in cu_seqlens]
    for a, b in zip(cu[:-1], cu[1:]):
        if b > a:
            out.append((a, b, float(np.linalg.norm(got[a:b] - ref[a:b])), float(np.linalg.norm(ref[a:b]))))
    return out


SHORT_SEGMENT = 16


def assert_per_segment(got: np.ndarray, ref: np.ndarray, cu_seqlens, tol: float, name: str) -> float:
    """The relative-L2 bound applied to every segment on its own, so that one
    wrong segment cannot hide in the norm of a whole tensor.  Returns the
    worst relative error over segments of at least SHORT_SEGMENT tokens.

    Shorter segments are held to the same bound on the larger of their own
    scale and the whole tensor's (RMS error <= tol x max(segment RMS, tensor
    RMS)): in a segment of a few tokens dq and dk are differences of nearly
    equal terms (each row of dS sums to zero), while the kernels take
    D = rowsum(dout * out) from the bf16-rounded out, whose error is relative
    to |dout| |out|, not to that difference.  A wrong segment still fails:
    its error is of the size of the values themselves.  A segment whose
    reference vanishes (length-1 segments, window 0: dS = 0 exactly) gets an
    absolute RMS bound of 1e-4."""
    worst = 0.0
    rms_all = float(np.sqrt(np.mean(np.square(ref))))
    for a, b, err, ref_norm in segment_errors(got, ref, cu_seqlens):
        n = ref[a:b].size
        if ref_norm < 1e-9:
            assert err / np.sqrt(n) <= 1e-4, (name, a, b, err)
            continue
        if b - a < SHORT_SEGMENT:
            scale = max(ref_norm / np.sqrt(n), rms_all)
            assert err / np.sqrt(n) <= tol * scale, (name, a, b, err / np.sqrt(n), scale)
            continue
        e = err / ref_norm
        worst = max(worst, e)
        assert e <= tol, (name, a, b, e)
    return worst


def to_device_bf16(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).to(device)


def run_gpu(inp, window_left: int, scale: float, max_seqlen: int, cu_override=None, backward: bool = True):
    """Runs fwd (+bwd) through the C ABI; returns numpy float64 arrays."""
    import torch
    from varlen_sliding_window_gb300 import binding
    dev = torch.device("cuda")
    q, k, v, do = (to_device_bf16(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits, inp.dout_bits))
    cu_np = inp.cu_seqlens if cu_override is None else cu_override
    cu = torch.from_numpy(np.asarray(cu_np, dtype=np.int32)).to(dev)
    T, hq = q.shape[0], q.shape[1]
    out = torch.full_like(q, float("nan"))
    lse = torch.full((hq, T), float("nan"), dtype=torch.float32, device=dev)
    binding.attn_varlen_fwd(q, k, v, cu, max_seqlen, window_left, scale, out, lse)
    res = {"out_t": out, "lse_t": lse}
    if backward:
        dq, dk, dv = (torch.full_like(x, float("nan")) for x in (q, k, v))
        binding.attn_varlen_bwd(do, q, k, v, out, lse, cu, max_seqlen, window_left, scale, dq, dk, dv)
        res.update(dq_t=dq, dk_t=dk, dv_t=dv)
    torch.cuda.synchronize()
    status = binding.attn_varlen_get_status()
    assert status == 0, f"device status word {status}"
    for name in list(res):
        res[name[:-2]] = res[name].double().cpu().numpy()
    return res


def segment_slice(inp, a: int, b: int):
    """The inputs of one segment as a standalone one-segment problem."""
    import copy
    sub = copy.copy(inp)
    for name in ("q", "k", "v", "dout"):
        setattr(sub, name, getattr(inp, name)[a:b])
    sub.cu_seqlens = np.array([0, b - a], dtype=np.int32)
    return sub


def by_key_ranges_from_oracle(cu_seqlens, window_left: int, total: int) -> np.ndarray:
    """For every key j: (first query seeing j, last query seeing j, count), from the oracle's masks."""
    import oracle
    out = np.zeros((total, 3), dtype=np.int64)
    out[:, 1] = -1
    for a, b in oracle.segments(cu_seqlens):
        L = b - a
        for r0 in range(0, L, 1024):
            r1 = min(L, r0 + 1024)
            m = oracle.visible_mask(a, b, window_left, r0, r1)  # [rows, L]
            cols = np.nonzero(m.any(axis=0))[0]
            for j in cols:
                rows = np.nonzero(m[:, j])[0] + r0
                if out[a + j, 2] == 0:
                    out[a + j, 0] = a + rows[0]
                out[a + j, 1] = a + rows[-1]
                out[a + j, 2] += rows.size
    return out
