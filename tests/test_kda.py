"""Kimi Delta attention on the GPU against the float64 oracle, through the C
ABI (include/kda_varlen.h).

Tolerance: relative L2 error <= 1.5e-2 over the whole tensor and over every
segment of at least 16 tokens (shorter ones: RMS error <= the bound x the
larger of their RMS and the tensor's).  On the way to o the kernels round to
bf16 the per-block scaled copies of K and Q that carry the per-channel decay
inside the products, the WY factors W and U, the masked q.k block, K o e^gamma,
Q o e^gamma, K o e^(gamma_last - gamma), the state copy used as an operand,
the pseudo-values E and o itself: about nine roundings of relative RMS
2^-8 / sqrt(3) = 2.3e-3, sqrt(9) x 2.3e-3 = 6.9e-3 together; the bound is
about twice that.  The gradients (relative L2 <= 2e-2 each, same per-segment
rule) add the recomputed factors, the bf16 copies of the state and of its
gradient, dE and dW, X as an operand and their outputs: about fifteen
roundings, sqrt(15) x 2.3e-3 = 8.9e-3, and again about twice that.
"""
import numpy as np
import pytest

from tests.helpers import assert_per_segment, rel_l2
from varlen_sliding_window_gb300 import synth

TOL_O = 1.5e-2
TOL_GRAD = 2e-2
WL = synth.kda_workloads()


def _to_dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).cuda()


def _run(inp, scale, cu=None):
    import torch
    from varlen_sliding_window_gb300 import binding
    cu = inp.cu_seqlens if cu is None else cu
    q, k, v = (_to_dev(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits))
    g = torch.from_numpy(inp.g).cuda()
    beta = torch.from_numpy(inp.beta).cuda()
    cu_t = torch.from_numpy(np.asarray(cu, dtype=np.int32)).cuda()
    T, nh, _ = q.shape
    o = torch.full_like(q, float("nan"))
    ws = torch.empty(binding.kda_varlen_workspace_bytes(T, nh, len(cu) - 1), dtype=torch.uint8, device="cuda")
    binding.kda_varlen_fwd(q, k, v, g, beta, cu_t, scale, o, ws)
    torch.cuda.synchronize()
    assert binding.attn_varlen_get_status() == 0
    return o


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["kda_tiny", "kda_ragged", "kda_ctx512", "kda_ctx4096"])
def test_forward_matches_oracle(name):
    from oracle import kimi_delta
    w = WL[name]
    inp = w.inputs()
    got = _run(inp, w.scale).double().cpu().numpy()
    ref = kimi_delta.forward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens, w.scale)
    assert np.isfinite(got).all()
    err = rel_l2(got, ref)
    print(f"{name}: rel L2 {err:.3e}")
    assert err <= TOL_O, err
    assert_per_segment(got, ref, inp.cu_seqlens, TOL_O, "o")


@pytest.mark.gpu
def test_equal_channels_match_the_gated_deltanet_kernels():
    # With the same gate on every channel the layer is Gated DeltaNet: the two
    # libraries' paths (different roundings) agree to the tolerance.
    import torch
    from varlen_sliding_window_gb300 import binding
    w = synth.gdn_workloads()["gdn_ragged"]
    inp = w.inputs()
    gk = np.ascontiguousarray(np.repeat(inp.g[:, :, None], w.d, axis=2))
    q, k, v = (_to_dev(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits))
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    T, nh = w.total, w.nh
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(max(binding.kda_varlen_workspace_bytes(T, nh, len(inp.cu_seqlens) - 1),
                         binding.gdn_varlen_workspace_bytes(T, nh, len(inp.cu_seqlens) - 1)), dtype=torch.uint8,
                     device="cuda")
    binding.kda_varlen_fwd(q, k, v, torch.from_numpy(gk).cuda(), torch.from_numpy(inp.beta).cuda(), cu, w.scale, o1,
                           ws)
    binding.gdn_varlen_fwd(q, k, v, torch.from_numpy(inp.g).cuda(), torch.from_numpy(inp.beta).cuda(), cu, w.scale,
                           o2, ws)
    torch.cuda.synchronize()
    assert rel_l2(o1.double().cpu().numpy(), o2.double().cpu().numpy()) <= TOL_O


@pytest.mark.gpu
def test_empty_segments_and_repeats_are_bit_identical():
    import torch
    w = WL["kda_ragged"]
    inp = w.inputs()
    a = _run(inp, w.scale)
    assert torch.equal(a, _run(inp, w.scale))
    cu = inp.cu_seqlens
    padded = np.concatenate([[0], cu[:4], cu[3:7], cu[6:], [cu[-1]] * 5]).astype(np.int32)
    assert torch.equal(a, _run(inp, w.scale, cu=padded))


def _run_bwd(inp, scale):
    import torch
    from varlen_sliding_window_gb300 import binding
    cu = inp.cu_seqlens
    q, k, v, do = (_to_dev(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    g = torch.from_numpy(inp.g).cuda()
    beta = torch.from_numpy(inp.beta).cuda()
    cu_t = torch.from_numpy(np.asarray(cu, dtype=np.int32)).cuda()
    T, nh, _ = q.shape
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    dg, dbeta = torch.full_like(g, float("nan")), torch.full_like(beta, float("nan"))
    ws = torch.empty(binding.kda_varlen_bwd_workspace_bytes(T, nh, len(cu) - 1), dtype=torch.uint8, device="cuda")
    binding.kda_varlen_bwd(q, k, v, g, beta, do, cu_t, scale, dq, dk, dv, dg, dbeta, ws)
    torch.cuda.synchronize()
    assert binding.attn_varlen_get_status() == 0
    return [x.double().cpu().numpy() for x in (dq, dk, dv, dg, dbeta)]


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["kda_tiny", "kda_ragged", "kda_ctx4096"])
def test_backward_matches_oracle(name):
    from oracle import kimi_delta
    w = WL[name]
    inp = w.inputs()
    got = _run_bwd(inp, w.scale)
    ref = kimi_delta.backward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.do, inp.cu_seqlens, w.scale)
    errs = {}
    for nm, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), got, ref):
        assert np.isfinite(a).all(), nm
        errs[nm] = rel_l2(a, b)
    print(name, {k: f"{v:.3e}" for k, v in errs.items()})
    for nm, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), got, ref):
        assert errs[nm] <= TOL_GRAD, (nm, errs[nm])
        assert_per_segment(a, b, inp.cu_seqlens, TOL_GRAD, nm)


@pytest.mark.gpu
def test_cuda_graph_replay_with_padded_boundaries_is_bit_exact():
    from tests.test_gdn import _graph_replay_is_bit_exact
    _graph_replay_is_bit_exact(synth.kda_workloads(), "kda_ctx4096", True)


@pytest.mark.gpu
def test_gate_at_or_below_the_bound_sets_the_status_word():
    """A log decay at or below -5.8 (the documented bound) is reported as
    ATTN_STATUS_GATE_RANGE (5) by the forward and by the backward; the same
    inputs with every gate clamped to -5.7 report nothing.  Out-of-range
    gates make no kernel fault or wait: the outputs are just not to be
    trusted."""
    import torch
    from varlen_sliding_window_gb300 import binding
    w = WL["kda_tiny"]
    inp = w.inputs()
    cu_t = torch.from_numpy(np.asarray(inp.cu_seqlens, dtype=np.int32)).cuda()
    q, k, v, do = (_to_dev(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    beta = torch.from_numpy(inp.beta).cuda()
    T, nh, _ = q.shape
    binding.attn_varlen_get_status()  # start from a clear word
    for bad in (True, False):
        g_np = np.maximum(inp.g, -5.7).astype(np.float32)
        if bad:
            g_np[T // 2, nh - 1, 77] = -6.0
        g = torch.from_numpy(g_np).cuda()
        o = torch.empty_like(q)
        ws = torch.empty(binding.kda_varlen_workspace_bytes(T, nh, len(inp.cu_seqlens) - 1), dtype=torch.uint8,
                         device="cuda")
        binding.kda_varlen_fwd(q, k, v, g, beta, cu_t, w.scale, o, ws)
        torch.cuda.synchronize()
        assert binding.attn_varlen_get_status() == (5 if bad else 0), ("fwd", bad)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        dg, dbeta = torch.empty_like(g), torch.empty_like(beta)
        wsb = torch.empty(binding.kda_varlen_bwd_workspace_bytes(T, nh, len(inp.cu_seqlens) - 1),
                          dtype=torch.uint8, device="cuda")
        binding.kda_varlen_bwd(q, k, v, g, beta, do, cu_t, w.scale, dq, dk, dv, dg, dbeta, wsb)
        torch.cuda.synchronize()
        assert binding.attn_varlen_get_status() == (5 if bad else 0), ("bwd", bad)


@pytest.mark.gpu
@pytest.mark.parametrize("nh", [1, 3, 5])
def test_head_counts(nh):
    from tests.test_gdn import check_head_counts
    check_head_counts(nh, per_channel=True)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["kda_ragged", "kda_ctx4096"])
def test_saving_forward_and_saved_backward_match_the_recomputing_pair(name):
    from tests.test_gdn import check_saved_pair
    check_saved_pair(WL, name, per_channel=True)
