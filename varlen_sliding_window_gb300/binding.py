"""Python binding of the C ABI in include/attn_varlen.h.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libvsw_attn.so.  Tensors are torch CUDA tensors (PyTorch is used
for device memory and streams).  There is no CPU fallback: if the library is
missing or the device is not an sm_103 GPU, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os

from ._build import LIB_PATH

_lib = None

ATTN_OK = 0


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = _strerror(code) if _lib is not None else str(code)
        super().__init__(f"{what} failed with {code}: {msg}")
        self.code = code


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Loads the in-tree library (built by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.attn_varlen_fwd.argtypes = [vp, vp, vp, vp, i32, i32, f32, vp, vp, i64, i32, i32, i32, i32, vp]
    lib.attn_varlen_fwd.restype = ctypes.c_int
    lib.attn_varlen_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, f32, vp, vp, vp, i64, i32, i32, i32, i32, vp]
    lib.attn_varlen_bwd.restype = ctypes.c_int
    lib.attn_varlen_bwd_workspace_bytes.argtypes = [i64, i32]
    lib.attn_varlen_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_varlen_workspace_bytes.argtypes = [i64, i32, i32, i32]
    lib.attn_varlen_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_varlen_set_workspace.argtypes = [vp, ctypes.c_size_t]
    lib.attn_varlen_set_workspace.restype = ctypes.c_int
    lib.attn_varlen_get_status.argtypes = [vp, ctypes.POINTER(i32)]
    lib.attn_varlen_get_status.restype = ctypes.c_int
    lib.attn_varlen_strerror.argtypes = [ctypes.c_int]
    lib.attn_varlen_strerror.restype = ctypes.c_char_p
    sz = ctypes.c_size_t
    lib.attn_varlen_bwd_preprocess.argtypes = [vp, vp, vp, sz, i64, i32, i32, vp]
    lib.attn_varlen_bwd_preprocess.restype = ctypes.c_int
    lib.attn_varlen_bwd_plan.argtypes = [vp, i32, i32, vp, sz, i64, i32, i32, i32, vp]
    lib.attn_varlen_bwd_plan.restype = ctypes.c_int
    lib.attn_varlen_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, sz, vp, i32, i32, f32, vp, vp, i64, i32, i32, i32, i32,
                                         vp]
    lib.attn_varlen_bwd_dkdv.restype = ctypes.c_int
    lib.attn_varlen_bwd_dq.argtypes = [vp, vp, vp, vp, vp, vp, sz, vp, i32, i32, f32, vp, i64, i32, i32, i32, i32, vp]
    lib.attn_varlen_bwd_dq.restype = ctypes.c_int
    lib.attn_varlen_fwd_strided.argtypes = lib.attn_varlen_fwd.argtypes[:-1] + [vp, vp]
    lib.attn_varlen_fwd_strided.restype = ctypes.c_int
    lib.attn_varlen_bwd_strided.argtypes = lib.attn_varlen_bwd.argtypes[:-1] + [vp, vp]
    lib.attn_varlen_bwd_strided.restype = ctypes.c_int
    lib.attn_varlen_bwd_noalloc.argtypes = lib.attn_varlen_bwd.argtypes
    lib.attn_varlen_bwd_noalloc.restype = ctypes.c_int
    lib.attn_varlen_mask_ranges.argtypes = [vp, i32, i64, i32, i32, i32, vp, vp]
    lib.attn_varlen_mask_ranges.restype = ctypes.c_int
    lib.gdn_varlen_workspace_bytes.argtypes = [i64, i32, i32]
    lib.gdn_varlen_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_varlen_fwd.argtypes = [vp, vp, vp, vp, vp, vp, f32, vp, vp, sz, i64, i32, i32, i32, vp]
    lib.gdn_varlen_fwd.restype = ctypes.c_int
    lib.gdn_varlen_bwd_workspace_bytes.argtypes = [i64, i32, i32]
    lib.gdn_varlen_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_varlen_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, f32, vp, vp, vp, vp, vp, vp, sz, i64, i32, i32, i32, vp]
    lib.gdn_varlen_bwd.restype = ctypes.c_int
    lib.kda_varlen_workspace_bytes.argtypes = [i64, i32, i32]
    lib.kda_varlen_workspace_bytes.restype = ctypes.c_size_t
    lib.kda_varlen_fwd.argtypes = lib.gdn_varlen_fwd.argtypes
    lib.kda_varlen_fwd.restype = ctypes.c_int
    lib.kda_varlen_bwd_workspace_bytes.argtypes = [i64, i32, i32]
    lib.kda_varlen_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.kda_varlen_bwd.argtypes = lib.gdn_varlen_bwd.argtypes
    lib.kda_varlen_bwd.restype = ctypes.c_int
    for name in ("gdn_varlen_fwd_save", "kda_varlen_fwd_save"):
        getattr(lib, name).argtypes = lib.gdn_varlen_fwd.argtypes
        getattr(lib, name).restype = ctypes.c_int
    for name in ("gdn_varlen_bwd_saved", "kda_varlen_bwd_saved"):
        getattr(lib, name).argtypes = lib.gdn_varlen_bwd.argtypes
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _strerror(code: int) -> str:
    return _lib.attn_varlen_strerror(code).decode()


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(code: int, what: str) -> None:
    if code != ATTN_OK:
        raise AttnError(code, what)


def _dims(q, k, cu_seqlens):
    total, hq, d = q.shape
    hkv = k.shape[1]
    return int(total), int(hq), int(hkv), int(d), int(cu_seqlens.numel()) - 1


def _strides(*tensors):
    """(token, head) element strides of [T, H, 128] views, as the int64 array the
    *_strided calls take; the last dimension must be contiguous."""
    vals = []
    for t in tensors:
        if t.dim() != 3 or t.stride(2) != 1:
            raise ValueError("expected a [T, H, 128] tensor with a contiguous last dimension")
        vals += [int(t.stride(0)), int(t.stride(1))]
    return (ctypes.c_int64 * len(vals))(*vals)


def _dense(*tensors) -> bool:
    return all(t.is_contiguous() for t in tensors)


def _require_dense(what: str, *tensors) -> None:
    """The calls without stride arguments read and write dense [T, H, 128] tensors."""
    if not _dense(*tensors):
        raise ValueError(f"{what} takes dense tensors; use the *_strided calls for views")


def _check_lse(lse):
    if not lse.is_contiguous():
        raise ValueError("lse must be a dense float32 [Hq, T] tensor")


def attn_varlen_fwd(q, k, v, cu_seqlens, max_seqlen: int, window_left: int, softmax_scale: float, out, lse,
                    stream=None) -> None:
    """Forward.  q [T,Hq,128], k/v [T,Hkv,128] bf16; out [T,Hq,128] bf16, lse [Hq,T] fp32.
    Strided views (last dimension contiguous) go through attn_varlen_fwd_strided."""
    if not _dense(q, k, v, out):
        return attn_varlen_fwd_strided(q, k, v, cu_seqlens, max_seqlen, window_left, softmax_scale, out, lse, stream)
    _check_lse(lse)
    lib = load_library()
    total, hq, hkv, d, nseg = _dims(q, k, cu_seqlens)
    rc = lib.attn_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), int(max_seqlen), int(window_left),
                             float(softmax_scale), _ptr(out), _ptr(lse), total, hq, hkv, d, nseg,
                             _stream_handle(stream))
    _check(rc, "attn_varlen_fwd")


def attn_varlen_fwd_strided(q, k, v, cu_seqlens, max_seqlen: int, window_left: int, softmax_scale: float, out, lse,
                            stream=None) -> None:
    """Forward on [T, H, 128] views with any 16-byte-multiple token/head strides."""
    _check_lse(lse)
    lib = load_library()
    total, hq, hkv, d, nseg = _dims(q, k, cu_seqlens)
    st = _strides(q, k, v, out)
    rc = lib.attn_varlen_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), int(max_seqlen), int(window_left),
                                     float(softmax_scale), _ptr(out), _ptr(lse), total, hq, hkv, d, nseg,
                                     ctypes.cast(st, ctypes.c_void_p), _stream_handle(stream))
    _check(rc, "attn_varlen_fwd_strided")


def attn_varlen_bwd(dout, q, k, v, out, lse, cu_seqlens, max_seqlen: int, window_left: int, softmax_scale: float,
                    dq, dk, dv, stream=None) -> None:
    """Backward.  Writes dq [T,Hq,128], dk/dv [T,Hkv,128] (bf16).  Strided views
    (last dimension contiguous) go through attn_varlen_bwd_strided."""
    if not _dense(dout, q, k, v, out, dq, dk, dv):
        return attn_varlen_bwd_strided(dout, q, k, v, out, lse, cu_seqlens, max_seqlen, window_left, softmax_scale,
                                       dq, dk, dv, stream)
    _check_lse(lse)
    lib = load_library()
    total, hq, hkv, d, nseg = _dims(q, k, cu_seqlens)
    rc = lib.attn_varlen_bwd(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens),
                             int(max_seqlen), int(window_left), float(softmax_scale), _ptr(dq), _ptr(dk), _ptr(dv),
                             total, hq, hkv, d, nseg, _stream_handle(stream))
    _check(rc, "attn_varlen_bwd")


def attn_varlen_bwd_strided(dout, q, k, v, out, lse, cu_seqlens, max_seqlen: int, window_left: int,
                            softmax_scale: float, dq, dk, dv, stream=None) -> None:
    """Backward on [T, H, 128] views with any 16-byte-multiple token/head strides."""
    _check_lse(lse)
    lib = load_library()
    total, hq, hkv, d, nseg = _dims(q, k, cu_seqlens)
    st = _strides(dout, q, k, v, out, dq, dk, dv)
    rc = lib.attn_varlen_bwd_strided(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens),
                                     int(max_seqlen), int(window_left), float(softmax_scale), _ptr(dq), _ptr(dk),
                                     _ptr(dv), total, hq, hkv, d, nseg, ctypes.cast(st, ctypes.c_void_p),
                                     _stream_handle(stream))
    _check(rc, "attn_varlen_bwd_strided")


def attn_varlen_bwd_noalloc(dout, q, k, v, out, lse, cu_seqlens, max_seqlen: int, window_left: int,
                            softmax_scale: float, dq, dk, dv, stream=None) -> None:
    """Backward with its scratch in the library's fixed device array (no allocation)."""
    _require_dense("attn_varlen_bwd_noalloc", dout, q, k, v, out, lse, dq, dk, dv)
    lib = load_library()
    total, hq, hkv, d, nseg = _dims(q, k, cu_seqlens)
    rc = lib.attn_varlen_bwd_noalloc(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens),
                                     int(max_seqlen), int(window_left), float(softmax_scale), _ptr(dq), _ptr(dk),
                                     _ptr(dv), total, hq, hkv, d, nseg, _stream_handle(stream))
    _check(rc, "attn_varlen_bwd_noalloc")


def _ws(workspace):
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def attn_varlen_bwd_preprocess(dout, out, workspace, stream=None) -> None:
    """D = rowsum(dout * out) into the workspace (a 256-byte-aligned uint8 CUDA tensor)."""
    _require_dense("attn_varlen_bwd_preprocess", dout, out)
    lib = load_library()
    total, hq, d = dout.shape
    wp, wb = _ws(workspace)
    _check(lib.attn_varlen_bwd_preprocess(_ptr(dout), _ptr(out), wp, wb, int(total), int(hq), int(d),
                                          _stream_handle(stream)), "attn_varlen_bwd_preprocess")


def attn_varlen_bwd_plan(cu_seqlens, max_seqlen: int, window_left: int, workspace, total: int, num_heads_q: int,
                         num_heads_kv: int, stream=None) -> None:
    """Writes the two passes' work lists into the workspace (optional sub-step)."""
    lib = load_library()
    wp, wb = _ws(workspace)
    _check(lib.attn_varlen_bwd_plan(_ptr(cu_seqlens), int(max_seqlen), int(window_left), wp, wb, int(total),
                                    int(num_heads_q), int(num_heads_kv), int(cu_seqlens.numel()) - 1,
                                    _stream_handle(stream)), "attn_varlen_bwd_plan")


def attn_varlen_bwd_dkdv(dout, q, k, v, lse, workspace, cu_seqlens, max_seqlen: int, window_left: int,
                         softmax_scale: float, dk, dv, stream=None) -> None:
    _require_dense("attn_varlen_bwd_dkdv", dout, q, k, v, lse, dk, dv)
    lib = load_library()
    total, hq, hkv, d, nseg = _dims(q, k, cu_seqlens)
    wp, wb = _ws(workspace)
    _check(lib.attn_varlen_bwd_dkdv(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(lse), wp, wb, _ptr(cu_seqlens),
                                    int(max_seqlen), int(window_left), float(softmax_scale), _ptr(dk), _ptr(dv),
                                    total, hq, hkv, d, nseg, _stream_handle(stream)), "attn_varlen_bwd_dkdv")


def attn_varlen_bwd_dq(dout, q, k, v, lse, workspace, cu_seqlens, max_seqlen: int, window_left: int,
                       softmax_scale: float, dq, stream=None) -> None:
    _require_dense("attn_varlen_bwd_dq", dout, q, k, v, lse, dq)
    lib = load_library()
    total, hq, hkv, d, nseg = _dims(q, k, cu_seqlens)
    wp, wb = _ws(workspace)
    _check(lib.attn_varlen_bwd_dq(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(lse), wp, wb, _ptr(cu_seqlens),
                                  int(max_seqlen), int(window_left), float(softmax_scale), _ptr(dq), total, hq, hkv,
                                  d, nseg, _stream_handle(stream)), "attn_varlen_bwd_dq")


def attn_varlen_bwd_workspace_bytes(total: int, num_heads_q: int) -> int:
    return int(load_library().attn_varlen_bwd_workspace_bytes(int(total), int(num_heads_q)))


def attn_varlen_workspace_bytes(total: int, num_heads_q: int, num_segments: int, max_seqlen: int) -> int:
    return int(load_library().attn_varlen_workspace_bytes(int(total), int(num_heads_q), int(num_segments),
                                                          int(max_seqlen)))


def attn_varlen_set_workspace(workspace) -> None:
    """Registers a caller-owned CUDA tensor (256-byte aligned) as the backward's
    scratch on the current device; None goes back to the library's own.  The
    caller keeps the tensor alive while calls that use it run."""
    lib = load_library()
    if workspace is None:
        _check(lib.attn_varlen_set_workspace(None, 0), "attn_varlen_set_workspace")
        return
    wp, wb = _ws(workspace)
    _check(lib.attn_varlen_set_workspace(wp, wb), "attn_varlen_set_workspace")


def attn_varlen_get_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status word."""
    lib = load_library()
    word = ctypes.c_int32(0)
    rc = lib.attn_varlen_get_status(_stream_handle(stream), ctypes.byref(word))
    if rc not in (ATTN_OK, -12):
        _check(rc, "attn_varlen_get_status")
    return int(word.value)


def attn_varlen_strerror(code: int) -> str:
    load_library()
    return _strerror(code)


def attn_varlen_mask_ranges(cu_seqlens, total: int, max_seqlen: int, window_left: int, by_key: bool, ranges,
                            stream=None) -> None:
    """Test hook: per-token (first, last, count) from the kernels' own mask logic."""
    lib = load_library()
    rc = lib.attn_varlen_mask_ranges(_ptr(cu_seqlens), int(cu_seqlens.numel()) - 1, int(total), int(max_seqlen),
                                     int(window_left), 1 if by_key else 0, _ptr(ranges), _stream_handle(stream))
    _check(rc, "attn_varlen_mask_ranges")


def default_scale(head_dim: int = 128) -> float:
    return 1.0 / math.sqrt(head_dim)


def gdn_varlen_workspace_bytes(total: int, num_heads: int, num_segments: int) -> int:
    """Device workspace bytes gdn_varlen_fwd needs (include/gdn_varlen.h)."""
    return int(load_library().gdn_varlen_workspace_bytes(int(total), int(num_heads), int(num_segments)))


def gdn_varlen_fwd(q, k, v, g, beta, cu_seqlens, scale: float, o, workspace, stream=None) -> None:
    """Gated DeltaNet forward over packed documents.  q, k, v, o: dense bf16
    [T, H, 128]; g, beta: dense float32 [T, H]; workspace: uint8 CUDA tensor of
    at least gdn_varlen_workspace_bytes(T, H, num_segments) bytes."""
    _require_dense("gdn_varlen_fwd", q, k, v, o)
    if not (g.is_contiguous() and beta.is_contiguous()):
        raise ValueError("g and beta must be dense float32 [T, H] tensors")
    lib = load_library()
    total, nh, d = (int(x) for x in q.shape)
    nseg = int(cu_seqlens.numel()) - 1
    rc = lib.gdn_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), float(scale), _ptr(o),
                            _ptr(workspace), int(workspace.numel()), total, nh, d, nseg, _stream_handle(stream))
    _check(rc, "gdn_varlen_fwd")


def gdn_varlen_bwd_workspace_bytes(total: int, num_heads: int, num_segments: int) -> int:
    """Device workspace bytes gdn_varlen_bwd needs (include/gdn_varlen.h)."""
    return int(load_library().gdn_varlen_bwd_workspace_bytes(int(total), int(num_heads), int(num_segments)))


def gdn_varlen_bwd(q, k, v, g, beta, d_o, cu_seqlens, scale: float, dq, dk, dv, dg, dbeta, workspace,
                   stream=None) -> None:
    """Gated DeltaNet backward: dq, dk, dv (bf16 [T, H, 128]) and dg, dbeta
    (float32 [T, H]) of sum(d_o * o); workspace of at least
    gdn_varlen_bwd_workspace_bytes(T, H, num_segments) bytes."""
    _require_dense("gdn_varlen_bwd", q, k, v, d_o, dq, dk, dv)
    for t in (g, beta, dg, dbeta):
        if not t.is_contiguous():
            raise ValueError("g, beta, dg and dbeta must be dense float32 [T, H] tensors")
    lib = load_library()
    total, nh, d = (int(x) for x in q.shape)
    nseg = int(cu_seqlens.numel()) - 1
    rc = lib.gdn_varlen_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(d_o), _ptr(cu_seqlens), float(scale),
                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(workspace),
                            int(workspace.numel()), total, nh, d, nseg, _stream_handle(stream))
    _check(rc, "gdn_varlen_bwd")


def kda_varlen_workspace_bytes(total: int, num_heads: int, num_segments: int) -> int:
    """Device workspace bytes kda_varlen_fwd needs (include/kda_varlen.h)."""
    return int(load_library().kda_varlen_workspace_bytes(int(total), int(num_heads), int(num_segments)))


def kda_varlen_fwd(q, k, v, g, beta, cu_seqlens, scale: float, o, workspace, stream=None) -> None:
    """Kimi Delta forward over packed documents.  q, k, v, o: dense bf16
    [T, H, 128]; g: dense float32 [T, H, 128] (log decay per key channel);
    beta: dense float32 [T, H]; workspace: uint8 CUDA tensor of at least
    kda_varlen_workspace_bytes(T, H, num_segments) bytes."""
    _require_dense("kda_varlen_fwd", q, k, v, o)
    if not (g.is_contiguous() and beta.is_contiguous()):
        raise ValueError("g and beta must be dense float32 tensors")
    lib = load_library()
    total, nh, d = (int(x) for x in q.shape)
    nseg = int(cu_seqlens.numel()) - 1
    rc = lib.kda_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), float(scale), _ptr(o),
                            _ptr(workspace), int(workspace.numel()), total, nh, d, nseg, _stream_handle(stream))
    _check(rc, "kda_varlen_fwd")


def kda_varlen_bwd_workspace_bytes(total: int, num_heads: int, num_segments: int) -> int:
    """Device workspace bytes kda_varlen_bwd needs (include/kda_varlen.h)."""
    return int(load_library().kda_varlen_bwd_workspace_bytes(int(total), int(num_heads), int(num_segments)))


def kda_varlen_bwd(q, k, v, g, beta, d_o, cu_seqlens, scale: float, dq, dk, dv, dg, dbeta, workspace,
                   stream=None) -> None:
    """Kimi Delta backward: dq, dk, dv (bf16 [T, H, 128]), dg (float32 [T, H, 128])
    and dbeta (float32 [T, H]) of sum(d_o * o)."""
    _require_dense("kda_varlen_bwd", q, k, v, d_o, dq, dk, dv)
    for t in (g, beta, dg, dbeta):
        if not t.is_contiguous():
            raise ValueError("g, beta, dg and dbeta must be dense float32 tensors")
    lib = load_library()
    total, nh, d = (int(x) for x in q.shape)
    nseg = int(cu_seqlens.numel()) - 1
    rc = lib.kda_varlen_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(d_o), _ptr(cu_seqlens), float(scale),
                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(workspace),
                            int(workspace.numel()), total, nh, d, nseg, _stream_handle(stream))
    _check(rc, "kda_varlen_bwd")


def _linear_fwd(name, q, k, v, g, beta, cu_seqlens, scale, o, workspace, stream):
    _require_dense(name, q, k, v, o)
    if not (g.is_contiguous() and beta.is_contiguous()):
        raise ValueError("g and beta must be dense float32 tensors")
    lib = load_library()
    total, nh, d = (int(x) for x in q.shape)
    nseg = int(cu_seqlens.numel()) - 1
    rc = getattr(lib, name)(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), float(scale), _ptr(o),
                            _ptr(workspace), int(workspace.numel()), total, nh, d, nseg, _stream_handle(stream))
    _check(rc, name)


def _linear_bwd(name, q, k, v, g, beta, d_o, cu_seqlens, scale, dq, dk, dv, dg, dbeta, workspace, stream):
    _require_dense(name, q, k, v, d_o, dq, dk, dv)
    for t in (g, beta, dg, dbeta):
        if not t.is_contiguous():
            raise ValueError("g, beta, dg and dbeta must be dense float32 tensors")
    lib = load_library()
    total, nh, d = (int(x) for x in q.shape)
    nseg = int(cu_seqlens.numel()) - 1
    rc = getattr(lib, name)(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(d_o), _ptr(cu_seqlens),
                            float(scale), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(workspace),
                            int(workspace.numel()), total, nh, d, nseg, _stream_handle(stream))
    _check(rc, name)


def gdn_varlen_fwd_save(q, k, v, g, beta, cu_seqlens, scale: float, o, workspace, stream=None) -> None:
    """gdn_varlen_fwd that also keeps what the backward recomputes in
    `workspace` (at least gdn_varlen_bwd_workspace_bytes(T, H, num_segments)
    bytes), for gdn_varlen_bwd_saved (include/gdn_varlen.h)."""
    _linear_fwd("gdn_varlen_fwd_save", q, k, v, g, beta, cu_seqlens, scale, o, workspace, stream)


def gdn_varlen_bwd_saved(q, k, v, g, beta, d_o, cu_seqlens, scale: float, dq, dk, dv, dg, dbeta, workspace,
                         stream=None) -> None:
    """gdn_varlen_bwd on the workspace of the preceding gdn_varlen_fwd_save
    with the same inputs: skips the recomputation, same bits."""
    _linear_bwd("gdn_varlen_bwd_saved", q, k, v, g, beta, d_o, cu_seqlens, scale, dq, dk, dv, dg, dbeta, workspace,
                stream)


def kda_varlen_fwd_save(q, k, v, g, beta, cu_seqlens, scale: float, o, workspace, stream=None) -> None:
    """kda_varlen_fwd that also keeps what the backward recomputes in
    `workspace` (at least kda_varlen_bwd_workspace_bytes(T, H, num_segments)
    bytes), for kda_varlen_bwd_saved (include/kda_varlen.h)."""
    _linear_fwd("kda_varlen_fwd_save", q, k, v, g, beta, cu_seqlens, scale, o, workspace, stream)


def kda_varlen_bwd_saved(q, k, v, g, beta, d_o, cu_seqlens, scale: float, dq, dk, dv, dg, dbeta, workspace,
                         stream=None) -> None:
    """kda_varlen_bwd on the workspace of the preceding kda_varlen_fwd_save
    with the same inputs: skips the recomputation, same bits."""
    _linear_bwd("kda_varlen_bwd_saved", q, k, v, g, beta, d_o, cu_seqlens, scale, dq, dk, dv, dg, dbeta, workspace,
                stream)
