"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function the header declares, and rejects invalid
arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_varlen.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))


@pytest.fixture(scope="module")
def clib():
    from varlen_sliding_window_gb300 import _build, binding
    _build.build_library()
    return binding.load_library()


def declared_functions():
    """Every function declared in include/*.h (comments stripped)."""
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b((?:attn|gdn|kda)_varlen_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_calls():
    names = declared_functions()
    for required in ("attn_varlen_fwd", "attn_varlen_bwd", "attn_varlen_get_status", "attn_varlen_strerror",
                     "gdn_varlen_fwd", "gdn_varlen_workspace_bytes", "gdn_varlen_bwd",
                     "gdn_varlen_bwd_workspace_bytes", "kda_varlen_fwd", "kda_varlen_workspace_bytes",
                     "kda_varlen_bwd", "kda_varlen_bwd_workspace_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol(clib):
    for name in declared_functions():
        assert hasattr(clib, name), name


def test_strerror(clib):
    assert clib.attn_varlen_strerror(0) == b"ok"
    assert b"128" in clib.attn_varlen_strerror(-3)
    assert clib.attn_varlen_strerror(12345) == b"unknown error code"


def _fwd(clib, **kw):
    args = dict(q=16, k=16, v=16, cu=16, max_seqlen=4, window=-1, scale=0.088, out=16, lse=16, total=4, hq=8,
                hkv=2, d=128, nseg=1, stream=None)
    args.update(kw)
    vp = ctypes.c_void_p
    return clib.attn_varlen_fwd(vp(args["q"]), vp(args["k"]), vp(args["v"]), vp(args["cu"]), args["max_seqlen"],
                                args["window"], args["scale"], vp(args["out"]), vp(args["lse"]), args["total"],
                                args["hq"], args["hkv"], args["d"], args["nseg"], vp(args["stream"]))


def test_argument_validation(clib):
    # All of these are rejected before any CUDA call, so no GPU is needed.
    assert _fwd(clib, q=None) == -1
    assert _fwd(clib, cu=None) == -1
    assert _fwd(clib, hq=6, hkv=4) == -2
    assert _fwd(clib, total=-1) == -2
    assert _fwd(clib, d=64) == -3
    assert _fwd(clib, q=17) == -4
    assert _fwd(clib, lse=20) == -4
    assert _fwd(clib, window=-2) == -5
    assert _fwd(clib, scale=float("nan")) == -6
    assert _fwd(clib, scale=0.0) == -6
    assert _fwd(clib, max_seqlen=5) == -7
    assert _fwd(clib, max_seqlen=-1) == -7


def test_strided_calls_check_their_strides(clib):
    # Rejected before any CUDA call: no GPU needed.
    vp = ctypes.c_void_p
    fake = vp(256)

    def fwd(strides):
        arr = None if strides is None else (ctypes.c_int64 * 8)(*strides)
        return clib.attn_varlen_fwd_strided(fake, fake, fake, fake, 4, -1, 0.088, fake, fake, 4, 8, 2, 128, 1,
                                            vp(None) if arr is None else ctypes.cast(arr, vp), vp(None))
    fused = [20 * 128, 128, 20 * 128, 128, 20 * 128, 128, 8 * 128, 128]  # q, k, v from one [T, 20, 128] buffer
    bad_cases = [
        [20 * 128, 100, 20 * 128, 128, 20 * 128, 128, 8 * 128, 128],  # head step below 128
        [20 * 128 + 4, 128, 20 * 128, 128, 20 * 128, 128, 8 * 128, 128],  # not a multiple of 8 elements
        [7 * 128, 128, 20 * 128, 128, 20 * 128, 128, 8 * 128, 128],  # token step below 8 heads x 128
        [0, 128, 20 * 128, 128, 20 * 128, 128, 8 * 128, 128],
        [20 * 128, 128, 20 * 128, 128, 20 * 128, 128, 8 * 128, -128],
    ]
    for bad in bad_cases:
        assert fwd(bad) == -15, bad
    assert fwd(None) == -1
    assert b"stride" in clib.attn_varlen_strerror(-15)
    # Valid strides get past the stride check (and fail later on the fake
    # pointers' alignment: 256 is aligned, so use a misaligned q instead).
    arr = (ctypes.c_int64 * 8)(*fused)
    rc = clib.attn_varlen_fwd_strided(vp(257), fake, fake, fake, 4, -1, 0.088, fake, fake, 4, 8, 2, 128, 1,
                                      ctypes.cast(arr, vp), vp(None))
    assert rc == -4


def test_workspace_bytes(clib):
    clib.attn_varlen_bwd_workspace_bytes.restype = ctypes.c_size_t
    clib.attn_varlen_bwd_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32]
    # counters, two run-time work lists of 32,768 36-byte items, 320 chain buffers
    chains = 2816 + 2 * 32768 * 36 + 320 * 2 * 128 * 128 * 4
    assert clib.attn_varlen_bwd_workspace_bytes(16384, 8) == 16384 * 8 * 4 + chains
    assert clib.attn_varlen_bwd_workspace_bytes(0, 8) == 0
    assert clib.attn_varlen_bwd_workspace_bytes(3, 1) == 256 + chains


def test_binding_fails_loudly_without_library(tmp_path):
    from varlen_sliding_window_gb300 import binding
    saved = binding._lib
    binding._lib = None
    try:
        with pytest.raises(RuntimeError, match="not built"):
            binding.load_library(str(tmp_path / "missing.so"))
    finally:
        binding._lib = saved


def test_binding_rejects_views_where_the_call_has_no_strides():
    import torch
    from varlen_sliding_window_gb300 import binding
    q = torch.zeros(4, 12, 128, dtype=torch.bfloat16)[:, :8]  # a view: token stride 12 * 128
    k = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    dense_q = torch.zeros(4, 8, 128, dtype=torch.bfloat16)
    lse = torch.zeros(8, 4)
    cu = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises(ValueError, match="strided"):
        binding.attn_varlen_bwd_noalloc(dense_q, q, k, k, dense_q, lse, cu, 4, -1, 0.088, dense_q, k, k)
    with pytest.raises(ValueError, match="strided"):
        binding.attn_varlen_bwd_preprocess(dense_q, q, torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(ValueError, match="lse"):
        binding.attn_varlen_fwd_strided(q, k, k, cu, 4, -1, 0.088, dense_q, lse.t())


def test_workspace_size_calls(clib):
    clib.attn_varlen_workspace_bytes.restype = ctypes.c_size_t
    clib.attn_varlen_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
    clib.attn_varlen_bwd_workspace_bytes.restype = ctypes.c_size_t
    clib.attn_varlen_bwd_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32]
    assert clib.attn_varlen_workspace_bytes(16384, 8, 25, 4096) == clib.attn_varlen_bwd_workspace_bytes(16384, 8)
    assert clib.attn_varlen_workspace_bytes(16384, 8, -1, 4096) == 0
    assert clib.attn_varlen_workspace_bytes(0, 8, 1, 0) == 0


def test_set_workspace_rejects_a_misaligned_buffer(clib):
    # The alignment check comes before the device probe: no GPU needed.
    clib.attn_varlen_set_workspace.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    assert clib.attn_varlen_set_workspace(ctypes.c_void_p(256 + 16), 1 << 20) == -4


def _gdn(clib, **kw):
    args = dict(q=16, k=16, v=16, g=16, beta=16, cu=16, scale=0.088, o=16, ws=256, ws_bytes=1 << 30, total=4, nh=8,
                d=128, nseg=1, stream=None)
    args.update(kw)
    vp = ctypes.c_void_p
    return clib.gdn_varlen_fwd(vp(args["q"]), vp(args["k"]), vp(args["v"]), vp(args["g"]), vp(args["beta"]),
                               vp(args["cu"]), args["scale"], vp(args["o"]), vp(args["ws"]), args["ws_bytes"],
                               args["total"], args["nh"], args["d"], args["nseg"], vp(args["stream"]))


def test_gdn_argument_validation(clib):
    # Rejected before any CUDA call, so no GPU is needed.
    assert _gdn(clib, q=None) == -1
    assert _gdn(clib, beta=None) == -1
    assert _gdn(clib, ws=None) == -1
    assert _gdn(clib, total=-1) == -2
    assert _gdn(clib, nh=0) == -2
    assert _gdn(clib, nseg=0) == -2
    assert _gdn(clib, d=64) == -3
    assert _gdn(clib, v=24) == -4
    assert _gdn(clib, g=20) == -4
    assert _gdn(clib, ws=272) == -4
    assert _gdn(clib, scale=float("inf")) == -6
    assert _gdn(clib, ws_bytes=1024) == -14


def test_gdn_workspace_bytes(clib):
    f = clib.gdn_varlen_workspace_bytes
    assert f(-1, 8, 1) == 0 and f(16, 0, 1) == 0
    n = f(16384, 8, 25)
    # W and U (bf16 [T, H, 128] each), the per-chunk q.k blocks, gamma and the tables
    assert n >= 2 * 16384 * 8 * 128 * 2 + (16384 // 64 + 25) * 8 * 64 * 64 * 2 + 16384 * 8 * 4
    assert n % 256 == 0
    assert f(16384, 8, 50) > n


def test_gdn_backward_argument_validation(clib):
    vp = ctypes.c_void_p

    def bwd(**kw):
        a = dict(q=16, k=16, v=16, g=16, beta=16, do=16, cu=16, dq=16, dk=16, dv=16, dg=16, db=16, ws=256,
                 ws_bytes=1 << 34, total=4, nh=8, d=128, nseg=1)
        a.update(kw)
        return clib.gdn_varlen_bwd(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]), vp(a["do"]),
                                   vp(a["cu"]), ctypes.c_float(0.088), vp(a["dq"]), vp(a["dk"]), vp(a["dv"]),
                                   vp(a["dg"]), vp(a["db"]), vp(a["ws"]), ctypes.c_size_t(a["ws_bytes"]),
                                   ctypes.c_int64(a["total"]), a["nh"], a["d"], a["nseg"], vp(None))
    assert bwd(do=None) == -1
    assert bwd(db=None) == -1
    assert bwd(d=64) == -3
    assert bwd(dk=40) == -4
    assert bwd(ws_bytes=4096) == -14
    f, fb = clib.gdn_varlen_workspace_bytes, clib.gdn_varlen_bwd_workspace_bytes
    assert fb(16384, 8, 25) > f(16384, 8, 25) > 0


def test_saving_forward_and_saved_backward_check_their_arguments(clib):
    # The saving forward keeps the backward's data: it needs the backward's
    # workspace size.  The saved backward checks what the backward checks.
    vp = ctypes.c_void_p
    for pre in ("gdn", "kda"):
        fwd_save = getattr(clib, f"{pre}_varlen_fwd_save")
        bwd_saved = getattr(clib, f"{pre}_varlen_bwd_saved")
        nf = getattr(clib, f"{pre}_varlen_workspace_bytes")(64, 8, 1)
        nb = getattr(clib, f"{pre}_varlen_bwd_workspace_bytes")(64, 8, 1)
        assert nb > nf > 0

        def fwd(ws_bytes, o=16, d=128):
            return fwd_save(vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), 0.088, vp(o), vp(256), ws_bytes, 64, 8, d,
                            1, vp(None))

        assert fwd(nf) == -14
        assert fwd(nb, o=None) == -1
        assert fwd(nb, d=64) == -3

        def bwd(ws_bytes, dq=16):
            return bwd_saved(vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), 0.088, vp(dq), vp(16), vp(16),
                             vp(16), vp(16), vp(256), ws_bytes, 64, 8, 128, 1, vp(None))

        assert bwd(nf) == -14
        assert bwd(nb, dq=None) == -1
        assert bwd(nb, dq=40) == -4
