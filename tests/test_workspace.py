"""The backward on a caller-registered workspace, and the status word for a
segment longer than max_seqlen (through the C ABI).

A training loop that replays a graph over fixed memory (research.dws.rip/
llm/kernels, section 06) registers its scratch once with
attn_varlen_set_workspace; attn_varlen_bwd then runs the same kernels, in the
same overlapped order, on that buffer.  With the full workspace size the
results are the same bits as on the library's own scratch; a buffer that
only holds D splits long key/value tiles less (other summation order, same
tolerance); a smaller one is refused.
"""
import numpy as np
import pytest

from varlen_sliding_window_gb300 import synth

from helpers import TOL_GRAD, rel_l2, to_device_bf16

pytestmark = pytest.mark.gpu

WL = synth.workloads()


def _setup(wl):
    import torch
    from varlen_sliding_window_gb300 import binding
    inp = wl.inputs()
    q, k, v, do = (to_device_bf16(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits, inp.dout_bits))
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    out = torch.empty_like(q)
    lse = torch.empty(wl.hq, wl.total, dtype=torch.float32, device="cuda")
    binding.attn_varlen_fwd(q, k, v, cu, wl.context, wl.window_left, wl.softmax_scale, out, lse)
    return q, k, v, do, cu, out, lse


def _bwd(wl, t):
    import torch
    from varlen_sliding_window_gb300 import binding
    q, k, v, do, cu, out, lse = t
    g = [torch.full_like(x, float("nan")) for x in (q, k, v)]
    binding.attn_varlen_bwd(do, q, k, v, out, lse, cu, wl.context, wl.window_left, wl.softmax_scale, *g)
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("name", ["ctx4096_global", "ctx4096_w512"])
def test_registered_workspace(name):
    import torch
    from varlen_sliding_window_gb300 import binding
    wl = WL[name]
    t = _setup(wl)
    binding.attn_varlen_get_status()
    ref = _bwd(wl, t)
    full = binding.attn_varlen_bwd_workspace_bytes(wl.total, wl.hq)
    assert full == binding.attn_varlen_workspace_bytes(wl.total, wl.hq, len(t[4]) - 1, wl.context)
    try:
        ws = torch.empty(full, dtype=torch.uint8, device="cuda")
        binding.attn_varlen_set_workspace(ws)
        for _ in range(2):  # twice: the second call sees what the first left in the buffer
            got = _bwd(wl, t)
            for nm, a, b in zip(("dq", "dk", "dv"), got, ref):
                assert torch.equal(a, b), nm
        # Room for D only: no split kv items, another summation order.
        small = torch.empty(wl.total * wl.hq * 4, dtype=torch.uint8, device="cuda")
        binding.attn_varlen_set_workspace(small)
        got = _bwd(wl, t)
        for nm, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(a.float()).all(), nm
            assert rel_l2(a.double().cpu().numpy(), b.double().cpu().numpy()) <= TOL_GRAD / 4, nm
        # Below the minimum: refused before anything is enqueued.
        binding.attn_varlen_set_workspace(small[: wl.total * wl.hq * 4 - 256])
        with pytest.raises(binding.AttnError) as e:
            _bwd(wl, t)
        assert e.value.code == -14
    finally:
        binding.attn_varlen_set_workspace(None)
    got = _bwd(wl, t)  # the library's own scratch again
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    assert binding.attn_varlen_get_status() == 0


def test_segment_longer_than_max_seqlen_is_reported():
    """max_seqlen below the longest segment: every kernel reports it through
    the status word (code 4); the right bound gives status 0."""
    import torch
    from varlen_sliding_window_gb300 import binding
    wl = WL["ctx4096_global"]
    q, k, v, do, cu, out, lse = _setup(wl)
    longest = int(np.diff(wl.cu_seqlens()).max())
    assert longest > 1024
    assert binding.attn_varlen_get_status() == 0
    binding.attn_varlen_fwd(q, k, v, cu, 1024, wl.window_left, wl.softmax_scale, out, lse)
    assert binding.attn_varlen_get_status() == 4
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    binding.attn_varlen_bwd(do, q, k, v, out, lse, cu, 1024, wl.window_left, wl.softmax_scale, dq, dk, dv)
    assert binding.attn_varlen_get_status() == 4
    # A bound that is not a tile multiple but still below the longest segment.
    binding.attn_varlen_fwd(q, k, v, cu, longest - 1, wl.window_left, wl.softmax_scale, out, lse)
    assert binding.attn_varlen_get_status() == 4
    binding.attn_varlen_fwd(q, k, v, cu, longest, wl.window_left, wl.softmax_scale, out, lse)
    binding.attn_varlen_bwd(do, q, k, v, out, lse, cu, longest, wl.window_left, wl.softmax_scale, dq, dk, dv)
    assert binding.attn_varlen_get_status() == 0


@pytest.mark.parametrize("name", ["ctx4096_global", "ctx512_global"])
def test_sub_step_calls_repeat_on_one_workspace(name):
    """The backward's kernels as separate calls on one caller workspace, the
    dK/dV and dQ passes each run four times after one preprocess, with and
    without a fresh plan: their run-time counters (split-item arrivals,
    claimed units) reset themselves, and claimed and fixed shares give the
    one-call backward's bits."""
    import torch
    from varlen_sliding_window_gb300 import binding
    wl = WL[name]
    q, k, v, do, cu, out, lse = t = _setup(wl)
    binding.attn_varlen_get_status()
    ref = _bwd(wl, t)
    ws = torch.empty(binding.attn_varlen_bwd_workspace_bytes(wl.total, wl.hq), dtype=torch.uint8, device="cuda")
    binding.attn_varlen_bwd_preprocess(do, out, ws)
    # With the work lists (claimed at run time), then twice without them
    # (each pass consumes its list and falls back to fixed shares), then with
    # a fresh plan again.
    for plan in (True, False, False, True):
        if plan:
            binding.attn_varlen_bwd_plan(cu, wl.context, wl.window_left, ws, wl.total, wl.hq, wl.hkv)
        dq, dk, dv = (torch.full_like(x, float("nan")) for x in (q, k, v))
        binding.attn_varlen_bwd_dkdv(do, q, k, v, lse, ws, cu, wl.context, wl.window_left, wl.softmax_scale, dk, dv)
        binding.attn_varlen_bwd_dq(do, q, k, v, lse, ws, cu, wl.context, wl.window_left, wl.softmax_scale, dq)
        torch.cuda.synchronize()
        for nm, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            assert torch.equal(a, b), (plan, nm)
    assert binding.attn_varlen_get_status() == 0
