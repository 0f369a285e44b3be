"""The no-allocation backward entry point.

attn_varlen_bwd_noalloc serves callers that may not allocate device memory
(code under an allocator it does not own or a fixed memory budget, real-time
callers for which an allocation may block or synchronise, paths that must
never call cudaMalloc).  It keeps its scratch in a fixed array inside the
library.  Here it is called through the C ABI twice in a row, on two
different microbatches, and each result is compared with attn_varlen_bwd on
the same inputs, within the gradient tolerance the other parity tests use.
Its size limit is checked too.

This file is collected last so that a run that stops at the first failure has
already run every other test; it does not depend on them.
"""
import ctypes

import numpy as np
import pytest

from varlen_sliding_window_gb300 import synth

from helpers import TOL_GRAD, rel_l2, to_device_bf16

pytestmark = pytest.mark.gpu


def _run_both(wl, cu):
    import torch
    from varlen_sliding_window_gb300 import binding
    inp = synth.make_inputs(cu, wl.hq, wl.hkv, wl.d, tensor_seed=wl.tensor_seed)
    q, k, v, do = (to_device_bf16(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits, inp.dout_bits))
    dcu = torch.from_numpy(np.asarray(cu, dtype=np.int32)).cuda()
    out = torch.empty_like(q)
    lse = torch.empty(wl.hq, q.shape[0], dtype=torch.float32, device="cuda")
    binding.attn_varlen_fwd(q, k, v, dcu, wl.context, wl.window_left, wl.softmax_scale, out, lse)
    ref = [torch.full_like(x, float("nan")) for x in (q, k, v)]
    binding.attn_varlen_bwd(do, q, k, v, out, lse, dcu, wl.context, wl.window_left, wl.softmax_scale, *ref)
    got = [torch.full_like(x, float("nan")) for x in (q, k, v)]
    binding.attn_varlen_bwd_noalloc(do, q, k, v, out, lse, dcu, wl.context, wl.window_left, wl.softmax_scale, *got)
    torch.cuda.synchronize()
    assert binding.attn_varlen_get_status() == 0
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g64, r64 = g.double().cpu().numpy(), r.double().cpu().numpy()
        assert np.all(np.isfinite(g64)), name
        assert rel_l2(g64, r64) <= TOL_GRAD, name


def test_noalloc_matches_allocating_backward_twice():
    wls = synth.workloads()
    # Two calls in a row on different microbatches and windows: the second
    # sees whatever the first left in the shared scratch.
    _run_both(wls["ctx4096_w512"], wls["ctx4096_w512"].cu_seqlens())
    _run_both(wls["ctx512_global"], wls["ctx512_global"].cu_seqlens())


def test_noalloc_rejects_problems_beyond_its_scratch():
    from varlen_sliding_window_gb300 import binding
    lib = binding.load_library()
    vp = ctypes.c_void_p
    fake = vp(256)  # never dereferenced: the size check comes first
    # T * Hq = 262,144 * 16 = 4,194,304 > 2,097,152
    rc = lib.attn_varlen_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, 4096, -1, 0.088, fake, fake, fake,
                                     262144, 16, 4, 128, 64, vp(None))
    assert rc == -13
    assert b"fixed scratch" in lib.attn_varlen_strerror(-13)
