"""The no-allocation backward entry point.

attn_varlen_bwd_noalloc serves callers that may not allocate device memory:
code under an allocator it does not own or a fixed memory budget, real-time
callers for which an allocation may block or synchronise the device, and
paths that must never call cudaMalloc.  It keeps its scratch in a fixed array
inside the library, with as many chain buffers as the allocating call uses,
so it runs the same kernels with the same work split and gives the same bits.

Here it is called through the C ABI on one microbatch, then twice in a row on
another (the array keeps whatever the call before left in it), and each
result must equal attn_varlen_bwd's bit for bit, with a clear status word.
On a smaller multi-tile case it is also compared with the float64 oracle, and
its size limit is checked.

This file is collected last so that a run that stops at the first failure has
already run every other test; it does not depend on them.
"""
import ctypes

import numpy as np
import pytest

import oracle
from varlen_sliding_window_gb300 import synth

from helpers import TOL_GRAD, assert_per_segment, rel_l2, to_device_bf16

pytestmark = pytest.mark.gpu


def _inputs(wl_or_cu, hq=8, hkv=2, seed=1):
    import torch
    if isinstance(wl_or_cu, np.ndarray):
        inp = synth.make_inputs(wl_or_cu, hq, hkv, 128, tensor_seed=seed)
    else:
        inp = wl_or_cu.inputs()
    q, k, v, do = (to_device_bf16(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits, inp.dout_bits))
    cu = torch.from_numpy(np.asarray(inp.cu_seqlens, dtype=np.int32)).cuda()
    return inp, (q, k, v, do, cu)


def _forward(t, max_seqlen, window, scale):
    import torch
    from varlen_sliding_window_gb300 import binding
    q, k, v, do, cu = t
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device="cuda")
    binding.attn_varlen_fwd(q, k, v, cu, max_seqlen, window, scale, out, lse)
    return out, lse


def _backward(fn, t, out, lse, max_seqlen, window, scale):
    import torch
    q, k, v, do, cu = t
    g = [torch.full_like(x, float("nan")) for x in (q, k, v)]
    fn(do, q, k, v, out, lse, cu, max_seqlen, window, scale, *g)
    torch.cuda.synchronize()
    return g


def test_noalloc_matches_allocating_backward_bitwise():
    import torch
    from varlen_sliding_window_gb300 import binding
    wls = synth.workloads()
    binding.attn_varlen_get_status()  # start from a clear status word
    results = []
    # A window-512 microbatch first, then the global one twice: its long kv
    # tiles are split into chains, whose buffers and counters live in the
    # shared array and carry over from the call before.
    for name in ("ctx4096_w512", "ctx4096_global", "ctx4096_global"):
        wl = wls[name]
        _, t = _inputs(wl)
        out, lse = _forward(t, wl.context, wl.window_left, wl.softmax_scale)
        ref = _backward(binding.attn_varlen_bwd, t, out, lse, wl.context, wl.window_left, wl.softmax_scale)
        got = _backward(binding.attn_varlen_bwd_noalloc, t, out, lse, wl.context, wl.window_left,
                        wl.softmax_scale)
        assert binding.attn_varlen_get_status() == 0, name
        for nm, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(a.float()).all(), (name, nm)
            assert torch.equal(a, b), (name, nm)
        results.append(got)
    for a, b in zip(results[1], results[2]):
        assert torch.equal(a, b)


def test_noalloc_against_the_oracle():
    """A ragged multi-tile case (segments of 1 to 513 tokens), compared with
    the float64 oracle element by element and per segment."""
    from varlen_sliding_window_gb300 import binding
    cu = np.array([0, 1, 130, 386, 387, 900, 1024, 1536, 1800], dtype=np.int32)
    scale = 1 / np.sqrt(128)
    for window in (-1, 300):
        inp, t = _inputs(cu, seed=3)
        out, lse = _forward(t, 600, window, scale)
        got = _backward(binding.attn_varlen_bwd_noalloc, t, out, lse, 600, window, scale)
        assert binding.attn_varlen_get_status() == 0
        ref = oracle.backward(inp.dout, inp.q, inp.k, inp.v, cu, window, scale)
        for nm, a, r in zip(("dq", "dk", "dv"), got, ref):
            a64 = a.double().cpu().numpy()
            assert rel_l2(a64, r) <= TOL_GRAD, (window, nm)
            assert_per_segment(a64, r, cu, TOL_GRAD, nm)


def test_noalloc_rejects_problems_beyond_its_scratch():
    from varlen_sliding_window_gb300 import binding
    lib = binding.load_library()
    vp = ctypes.c_void_p
    fake = vp(256)  # never dereferenced: the size check comes before anything is enqueued
    # T * Hq = 262,144 * 16 = 4,194,304 > 2,097,152
    rc = lib.attn_varlen_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, 4096, -1, 0.088, fake, fake, fake,
                                     262144, 16, 4, 128, 64, vp(None))
    assert rc == -13
    assert b"fixed scratch" in lib.attn_varlen_strerror(-13)
