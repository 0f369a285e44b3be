"""Seeded synthetic inputs: packed document microbatches and bf16 tensors.

This module holds no attention arithmetic.  It is the one piece that the CUDA
path's tests/benchmark and the CPU oracle both consume: it produces segment
boundaries (``cu_seqlens``) and bf16-representable q/k/v/dout values.

Workload recipe (research.dws.rip/llm/kernels, section 01 "How it was
measured", and Fig. 2 "Benchmark setup"): a microbatch is 16,384 tokens of
documents whose median length is 457 tokens while 45 % of all tokens sit in
documents of 4,096 tokens or more.  No document attends across its boundary
and each row is cut at the context length (512 ... 4,096), so a kernel sees a
few dozen segments.  The real token shards are not available; a log-normal
length law with median 457 and sigma 1.42 reproduces both statistics the page
gives (median 457, token share of >=4,096-token documents ~0.45).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

DOC_MEDIAN = 457.0
DOC_SIGMA = 1.42


def draw_document_lengths(total_tokens: int, doc_seed: int, cap: int | None = None) -> list[int]:
    """Draws document lengths one at a time until they cover ``total_tokens``."""
    rng = np.random.default_rng(doc_seed)
    lengths: list[int] = []
    acc = 0
    mu = math.log(DOC_MEDIAN)
    while acc < total_tokens:
        L = max(1, int(round(float(rng.lognormal(mu, DOC_SIGMA)))))
        if cap is not None:
            L = min(L, cap)
        lengths.append(L)
        acc += L
    return lengths


def pack_microbatch(total_tokens: int, context: int, doc_seed: int, cap: int | None = None) -> np.ndarray:
    """Packs documents end to end into rows of ``context`` tokens.

    Segment boundaries are the document ends, the row ends (multiples of
    ``context``) and {0, total}.  Returns ``cu_seqlens`` as int32 [nseg+1].
    """
    lengths = draw_document_lengths(total_tokens, doc_seed, cap)
    ends = np.cumsum(np.asarray(lengths, dtype=np.int64))
    bounds = set(int(e) for e in ends if e < total_tokens)
    bounds.update(range(0, total_tokens + 1, context))
    bounds.add(0)
    bounds.add(total_tokens)
    return np.asarray(sorted(bounds), dtype=np.int32)


def pad_cu_seqlens(cu_seqlens: np.ndarray, num_segments: int) -> np.ndarray:
    """Pads a boundary list with empty segments up to ``num_segments`` segments.

    Fixed-size boundary lists keep shapes constant for CUDA-graph replay
    (research.dws.rip/llm/kernels, section 06 and Fig. 8: padded to 42).
    """
    cu = np.asarray(cu_seqlens, dtype=np.int32)
    nseg = cu.size - 1
    if num_segments < nseg:
        raise ValueError("cannot pad to fewer segments than present")
    pad = np.full(num_segments - nseg, cu[-1], dtype=np.int32)
    return np.concatenate([cu, pad])


def round_to_bf16(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Rounds float32 values to bf16 (nearest, ties to even).

    Returns (bits uint16, values float32) where the float32 values are exactly
    the bf16 numbers.  Inputs are finite.
    """
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    bits = rounded.astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    return bits, vals


@dataclasses.dataclass
class Inputs:
    cu_seqlens: np.ndarray  # int32 [nseg+1]
    q: np.ndarray           # float32 (bf16 values) [T, Hq, d]
    k: np.ndarray           # float32 (bf16 values) [T, Hkv, d]
    v: np.ndarray
    dout: np.ndarray        # float32 (bf16 values) [T, Hq, d]
    q_bits: np.ndarray      # uint16 bf16 bit patterns, same shapes
    k_bits: np.ndarray
    v_bits: np.ndarray
    dout_bits: np.ndarray


def make_tensors(total: int, hq: int, hkv: int, d: int, tensor_seed: int) -> dict[str, tuple[np.ndarray, np.ndarray]]:
    """Draws q, k, v, dout (in that order) as N(0,1) float32, rounded to bf16."""
    rng = np.random.default_rng(tensor_seed)
    out = {}
    for name, h in (("q", hq), ("k", hkv), ("v", hkv), ("dout", hq)):
        x = rng.standard_normal((total, h, d), dtype=np.float32)
        out[name] = round_to_bf16(x)
    return out


def make_inputs(cu_seqlens: np.ndarray, hq: int, hkv: int, d: int, tensor_seed: int) -> Inputs:
    total = int(cu_seqlens[-1])
    t = make_tensors(total, hq, hkv, d, tensor_seed)
    return Inputs(cu_seqlens=np.asarray(cu_seqlens, dtype=np.int32),
                  q=t["q"][1], k=t["k"][1], v=t["v"][1], dout=t["dout"][1],
                  q_bits=t["q"][0], k_bits=t["k"][0], v_bits=t["v"][0], dout_bits=t["dout"][0])


@dataclasses.dataclass(frozen=True)
class Workload:
    """One named workload: shapes, window and seeds."""
    name: str
    total: int
    context: int
    window_left: int          # -1 = global causal
    hq: int = 8
    hkv: int = 2
    d: int = 128
    cap: int | None = None
    doc_seed: int = 0
    tensor_seed: int = 1
    fixed_cu: tuple[int, ...] | None = None

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def cu_seqlens(self) -> np.ndarray:
        if self.fixed_cu is not None:
            return np.asarray(self.fixed_cu, dtype=np.int32)
        return pack_microbatch(self.total, self.context, self.doc_seed, self.cap)

    def inputs(self) -> Inputs:
        return make_inputs(self.cu_seqlens(), self.hq, self.hkv, self.d, self.tensor_seed)


def workloads() -> dict[str, Workload]:
    """The named workloads: the 256-token three-document check, the
    16,384-token microbatches at context 512 and 4,096 (global and window 512),
    the context sweep, and the 65,536-token long-context case, global and with
    a 4,096-token window."""
    w: dict[str, Workload] = {}
    for win, tag in ((-1, "global"), (64, "w64")):
        w[f"tiny_{tag}"] = Workload(f"tiny_{tag}", 256, 256, win, tensor_seed=0, fixed_cu=(0, 61, 161, 256))
    w["ctx512_global"] = Workload("ctx512_global", 16384, 512, -1)
    w["ctx4096_w512"] = Workload("ctx4096_w512", 16384, 4096, 512)
    w["ctx4096_global"] = Workload("ctx4096_global", 16384, 4096, -1)
    for ctx in (512, 1024, 2048, 4096):
        for win, tag in ((-1, "global"), (512, "w512")):
            name = f"sweep_ctx{ctx}_{tag}"
            w[name] = Workload(name, 16384, ctx, win)
    w["long65536_global"] = Workload("long65536_global", 65536, 32768, -1, hq=16, hkv=4, cap=32768)
    # The same long microbatch with a 4,096-token window (the packed
    # sliding-window benchmark of dewml.dev/reference/performance).
    w["long65536_w4096"] = Workload("long65536_w4096", 65536, 32768, 4096, hq=16, hkv=4, cap=32768)
    return w


# ---------------------------------------------------------------- Gated DeltaNet
@dataclasses.dataclass
class GdnInputs:
    cu_seqlens: np.ndarray  # int32 [nseg+1]
    q: np.ndarray           # float32 (bf16 values) [T, H, d], rows of unit L2 norm before rounding
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray          # float32 (bf16 values) [T, H, d]
    g: np.ndarray           # float32 [T, H], log decay
    beta: np.ndarray        # float32 [T, H]
    q_bits: np.ndarray
    k_bits: np.ndarray
    v_bits: np.ndarray
    do_bits: np.ndarray


def make_gdn_inputs(cu_seqlens: np.ndarray, nh: int, d: int, tensor_seed: int,
                    per_channel: bool = False) -> GdnInputs:
    """Inputs of the Gated DeltaNet (or, with per_channel, Kimi Delta) local
    layer on a packed microbatch.  Drawn from default_rng(tensor_seed) in this
    order: q, k, v, do as N(0,1) float32 [T, H, d]; q and k rows divided by
    their L2 norm (the layer normalises them before the kernel); all four
    rounded to bf16; then g = -softplus(x), x ~ N(-5, 1.5) (decays exp(g)
    mostly 0.9 to 0.9995: long memory), float32 [T, H], or [T, H, d] with a
    gate per key channel; and beta = sigmoid(y), y ~ N(0, 1), float32 [T, H]."""
    cu = np.asarray(cu_seqlens, dtype=np.int32)
    total = int(cu[-1])
    rng = np.random.default_rng(tensor_seed)
    draws = {}
    for name in ("q", "k", "v", "do"):
        x = rng.standard_normal((total, nh, d), dtype=np.float32)
        if name in ("q", "k"):
            x = x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), np.float32(1e-6))
        draws[name] = round_to_bf16(x)
    x = rng.normal(-5.0, 1.5, size=(total, nh, d) if per_channel else (total, nh)).astype(np.float32)
    g = (-np.logaddexp(np.float32(0.0), x)).astype(np.float32)
    y = rng.standard_normal((total, nh), dtype=np.float32)
    beta = (1.0 / (1.0 + np.exp(-y))).astype(np.float32)
    return GdnInputs(cu_seqlens=cu, q=draws["q"][1], k=draws["k"][1], v=draws["v"][1], do=draws["do"][1], g=g,
                     beta=beta, q_bits=draws["q"][0], k_bits=draws["k"][0], v_bits=draws["v"][0],
                     do_bits=draws["do"][0])


@dataclasses.dataclass(frozen=True)
class GdnWorkload:
    """The Gated DeltaNet layer on one of the packed microbatches above
    (research.dws.rip/llm/kernels, section 03: same microbatches, 8 heads of
    width 128)."""
    name: str
    total: int
    context: int
    nh: int = 8
    d: int = 128
    doc_seed: int = 0
    tensor_seed: int = 1
    fixed_cu: tuple[int, ...] | None = None
    per_channel: bool = False  # Kimi Delta: a decay per key channel

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def cu_seqlens(self) -> np.ndarray:
        if self.fixed_cu is not None:
            return np.asarray(self.fixed_cu, dtype=np.int32)
        return pack_microbatch(self.total, self.context, self.doc_seed)

    def inputs(self) -> GdnInputs:
        return make_gdn_inputs(self.cu_seqlens(), self.nh, self.d, self.tensor_seed, self.per_channel)


def gdn_workloads() -> dict[str, GdnWorkload]:
    """The 256-token three-document check (seeds as the attention one), a
    ragged case whose segments end just before, at and after chunk edges, and
    the 16,384-token microbatches at context 4,096 and 512."""
    w: dict[str, GdnWorkload] = {}
    w["gdn_tiny"] = GdnWorkload("gdn_tiny", 256, 256, tensor_seed=0, fixed_cu=(0, 61, 161, 256))
    lens = (1, 63, 64, 65, 0, 127, 128, 129, 200, 0, 2, 300)
    cu = tuple(int(x) for x in np.concatenate([[0], np.cumsum(lens)]))
    w["gdn_ragged"] = GdnWorkload("gdn_ragged", cu[-1], 512, nh=4, tensor_seed=3, fixed_cu=cu)
    w["gdn_ctx4096"] = GdnWorkload("gdn_ctx4096", 16384, 4096)
    w["gdn_ctx512"] = GdnWorkload("gdn_ctx512", 16384, 512)
    return w


def kda_workloads() -> dict[str, GdnWorkload]:
    """The Kimi Delta layer on the same cases as gdn_workloads(), with a gate
    per key channel."""
    import dataclasses
    return {n.replace("gdn_", "kda_"): dataclasses.replace(w, name=w.name.replace("gdn_", "kda_"), per_channel=True)
            for n, w in gdn_workloads().items()}
