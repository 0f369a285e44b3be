"""Gated DeltaNet forward on the GPU against the float64 oracle, through the
C ABI (include/gdn_varlen.h).

Tolerance: relative L2 error of o <= 1e-2 over the whole tensor and over
every segment of at least 16 tokens (shorter ones: RMS error <= 1e-2 x the
larger of their RMS and the tensor's).  The kernels round to bf16, on the
way to each output, the WY factors W and U, the masked q.k block, the state
copy used as a matrix operand, the pseudo-values E, and o itself: six
roundings, each with a relative RMS error of about 2^-8 / sqrt(3) = 2.3e-3;
independent, they add up to sqrt(6) x 2.3e-3 = 5.5e-3.  The bound is about
twice that.  (The oracle sees the same bf16 q, k, v and float32 g, beta.)
The gradients (dq, dk, dv, dg, dbeta; relative L2 <= 1.5e-2 each, same
per-segment rule) pass through about eight such roundings (the recomputed
factors, the bf16 copies of the state and of its gradient, dE, dW, the
masked blocks DG and M, X as an operand, and the output):
sqrt(8) x 2.3e-3 = 6.5e-3, and the bound is again about twice that.
"""
import numpy as np
import pytest

from tests.helpers import assert_per_segment, rel_l2
from varlen_sliding_window_gb300 import synth

TOL_O = 1e-2
TOL_GRAD = {"dq": 1.5e-2, "dk": 1.5e-2, "dv": 1.5e-2, "dg": 1.5e-2, "dbeta": 1.5e-2}
WL = synth.gdn_workloads()


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
    ws = torch.empty(binding.gdn_varlen_workspace_bytes(T, nh, len(cu) - 1), dtype=torch.uint8, device="cuda")
    binding.gdn_varlen_fwd(q, k, v, g, beta, cu_t, scale, o, ws)
    torch.cuda.synchronize()
    assert binding.attn_varlen_get_status() == 0
    return o


def _oracle(inp, scale):
    from oracle import gated_delta
    return gated_delta.forward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens, scale)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["gdn_tiny", "gdn_ragged", "gdn_ctx512", "gdn_ctx4096"])
def test_forward_matches_oracle(name):
    w = WL[name]
    inp = w.inputs()
    got = _run(inp, w.scale).double().cpu().numpy()
    ref = _oracle(inp, w.scale)
    assert np.isfinite(got).all()
    err = rel_l2(got, ref)
    print(f"{name}: rel L2 {err:.3e}")
    assert err <= TOL_O, err
    assert_per_segment(got, ref, inp.cu_seqlens, TOL_O, "o")


@pytest.mark.gpu
def test_empty_segments_and_repeats_are_bit_identical():
    import torch
    w = WL["gdn_ragged"]
    inp = w.inputs()
    a = _run(inp, w.scale)
    b = _run(inp, w.scale)
    assert torch.equal(a, b)
    cu = inp.cu_seqlens
    padded = np.concatenate([[0], cu[:4], cu[3:7], cu[6:], [cu[-1]] * 5]).astype(np.int32)
    assert np.all(np.diff(padded) >= 0) and padded[-1] == cu[-1]
    c = _run(inp, w.scale, cu=padded)
    assert torch.equal(a, c)


@pytest.mark.gpu
def test_segments_do_not_share_state():
    # One document's inputs changed: every other document's outputs keep their bits.
    import torch
    w = WL["gdn_ragged"]
    inp = w.inputs()
    a = _run(inp, w.scale)
    cu = inp.cu_seqlens
    lo, hi = int(cu[5]), int(cu[6])  # the 127-token segment
    inp2 = synth.make_gdn_inputs(cu, w.nh, w.d, w.tensor_seed)
    inp2.v_bits = inp2.v_bits.copy()
    inp2.v_bits[lo:hi] ^= np.uint16(0x0040)
    inp2.g = inp2.g.copy()
    inp2.g[lo:hi] *= 0.5
    b = _run(inp2, w.scale)
    assert not torch.equal(a[lo:hi], b[lo:hi])
    assert torch.equal(a[:lo], b[:lo]) and torch.equal(a[hi:], b[hi:])


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
    dg, dbeta = (torch.full_like(g, float("nan")) for _ in range(2))
    ws = torch.empty(binding.gdn_varlen_bwd_workspace_bytes(T, nh, len(cu) - 1), dtype=torch.uint8, device="cuda")
    binding.gdn_varlen_bwd(q, k, v, g, beta, do, cu_t, scale, dq, dk, dv, dg, dbeta, ws)
    torch.cuda.synchronize()
    assert binding.attn_varlen_get_status() == 0
    return [x.double().cpu().numpy() for x in (dq, dk, dv, dg, dbeta)]


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["gdn_tiny", "gdn_ragged", "gdn_ctx4096"])
def test_backward_matches_oracle(name):
    from oracle import gated_delta
    w = WL[name]
    inp = w.inputs()
    got = _run_bwd(inp, w.scale)
    ref = gated_delta.backward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.do, inp.cu_seqlens, w.scale)
    errs = {}
    for nm, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), got, ref):
        assert np.isfinite(a).all(), nm
        errs[nm] = rel_l2(a, b)
    print(name, {k: f"{v:.3e}" for k, v in errs.items()})
    for nm, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), got, ref):
        assert errs[nm] <= TOL_GRAD[nm], (nm, errs[nm])
        assert_per_segment(a, b, inp.cu_seqlens, TOL_GRAD[nm], nm)


def _graph_replay_is_bit_exact(wls, name, per_channel):
    """Forward + backward captured once in a CUDA graph over a boundary list
    padded with empty segments to 42 (research.dws.rip/llm/kernels, section
    06), replayed on three microbatches with different boundaries: every output
    bit-equal to eager calls on the unpadded boundaries."""
    import torch
    from varlen_sliding_window_gb300 import binding
    w = wls[name]
    f_fwd, f_bwd, f_ws = ((binding.kda_varlen_fwd, binding.kda_varlen_bwd, binding.kda_varlen_bwd_workspace_bytes)
                          if per_channel else
                          (binding.gdn_varlen_fwd, binding.gdn_varlen_bwd, binding.gdn_varlen_bwd_workspace_bytes))
    cus = [synth.pack_microbatch(w.total, w.context, sd) for sd in (0, 1, 2)]
    nseg = 42
    assert max(len(c) - 1 for c in cus) <= nseg
    batches = [synth.make_gdn_inputs(c, w.nh, w.d, 10 + i, per_channel) for i, c in enumerate(cus)]
    T, nh = w.total, w.nh
    st = {"q": torch.empty(T, nh, w.d, dtype=torch.bfloat16, device="cuda")}
    for n in ("k", "v", "do", "o", "dq", "dk", "dv"):
        st[n] = torch.empty_like(st["q"])
    gshape = (T, nh, w.d) if per_channel else (T, nh)
    for n in ("g", "dg"):
        st[n] = torch.empty(gshape, dtype=torch.float32, device="cuda")
    for n in ("beta", "dbeta"):
        st[n] = torch.empty(T, nh, dtype=torch.float32, device="cuda")
    st["cu"] = torch.empty(nseg + 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(f_ws(T, nh, nseg), dtype=torch.uint8, device="cuda")

    def load(b, cu):
        for n, bits in (("q", b.q_bits), ("k", b.k_bits), ("v", b.v_bits), ("do", b.do_bits)):
            st[n].copy_(_to_dev(bits))
        st["g"].copy_(torch.from_numpy(b.g))
        st["beta"].copy_(torch.from_numpy(b.beta))
        st["cu"].copy_(torch.from_numpy(synth.pad_cu_seqlens(cu, nseg)))

    def step():
        f_fwd(st["q"], st["k"], st["v"], st["g"], st["beta"], st["cu"], w.scale, st["o"], ws)
        f_bwd(st["q"], st["k"], st["v"], st["g"], st["beta"], st["do"], st["cu"], w.scale, st["dq"], st["dk"],
              st["dv"], st["dg"], st["dbeta"], ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    load(batches[0], cus[0])
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step()
    names = ("o", "dq", "dk", "dv", "dg", "dbeta")
    for b, cu in zip(batches, cus):
        load(b, cu)
        graph.replay()
        torch.cuda.synchronize()
        got = {n: st[n].clone() for n in names}
        # eager, unpadded boundaries, own buffers
        e = {n: torch.empty_like(st[n]) for n in names}
        cu_t = torch.from_numpy(cu).cuda()
        ws2 = torch.empty(f_ws(T, nh, len(cu) - 1), dtype=torch.uint8, device="cuda")
        f_fwd(st["q"], st["k"], st["v"], st["g"], st["beta"], cu_t, w.scale, e["o"], ws2)
        f_bwd(st["q"], st["k"], st["v"], st["g"], st["beta"], st["do"], cu_t, w.scale, e["dq"], e["dk"], e["dv"],
              e["dg"], e["dbeta"], ws2)
        torch.cuda.synchronize()
        for n in names:
            assert torch.equal(got[n], e[n]), n
    from varlen_sliding_window_gb300 import binding as _b
    assert _b.attn_varlen_get_status() == 0


@pytest.mark.gpu
def test_cuda_graph_replay_with_padded_boundaries_is_bit_exact():
    _graph_replay_is_bit_exact(synth.gdn_workloads(), "gdn_ctx4096", False)


def check_saved_pair(wls, name, per_channel):
    """The saving forward and the backward on its workspace
    (include/gdn_varlen.h, include/kda_varlen.h) give the bits of the
    recomputing pair: o, dq, dk, dv, dg, dbeta all equal, also when the
    saved pair runs twice on one workspace."""
    import torch
    from varlen_sliding_window_gb300 import binding as b
    w = wls[name]
    inp = w.inputs()
    pre = "kda" if per_channel else "gdn"
    fwd, bwd = getattr(b, f"{pre}_varlen_fwd"), getattr(b, f"{pre}_varlen_bwd")
    fwd_save, bwd_saved = getattr(b, f"{pre}_varlen_fwd_save"), getattr(b, f"{pre}_varlen_bwd_saved")
    ws_f, ws_b = getattr(b, f"{pre}_varlen_workspace_bytes"), getattr(b, f"{pre}_varlen_bwd_workspace_bytes")
    q, k, v, do = (_to_dev(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    g = torch.from_numpy(inp.g).cuda()
    beta = torch.from_numpy(inp.beta).cuda()
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    T, nh, _ = q.shape
    nseg = len(inp.cu_seqlens) - 1

    def outs():
        o = torch.full_like(q, float("nan"))
        grads = [torch.full_like(q, float("nan")) for _ in range(3)] + [torch.full_like(g, float("nan")),
                                                                         torch.full_like(beta, float("nan"))]
        return o, grads

    o1, g1 = outs()
    wf = torch.empty(ws_f(T, nh, nseg), dtype=torch.uint8, device="cuda")
    wb = torch.empty(ws_b(T, nh, nseg), dtype=torch.uint8, device="cuda")
    fwd(q, k, v, g, beta, cu, w.scale, o1, wf)
    bwd(q, k, v, g, beta, do, cu, w.scale, *g1, wb)
    ws = torch.empty(ws_b(T, nh, nseg), dtype=torch.uint8, device="cuda")
    for _ in range(2):
        o2, g2 = outs()
        fwd_save(q, k, v, g, beta, cu, w.scale, o2, ws)
        bwd_saved(q, k, v, g, beta, do, cu, w.scale, *g2, ws)
        torch.cuda.synchronize()
        assert b.attn_varlen_get_status() == 0
        assert torch.equal(o1, o2)
        for nm, a, c in zip(("dq", "dk", "dv", "dg", "dbeta"), g1, g2):
            assert torch.equal(a, c), nm


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["gdn_ragged", "gdn_ctx4096"])
def test_saving_forward_and_saved_backward_match_the_recomputing_pair(name):
    check_saved_pair(WL, name, per_channel=False)


# Ragged boundaries for the head-count cases: a 1-token segment, segments
# ending one before, at and one after a 64-token chunk edge, an empty one.
HEAD_CASE_CU = np.array([0, 1, 64, 65, 129, 129, 200, 330], dtype=np.int32)


def check_head_counts(nh, per_channel):
    """Forward and backward against the oracle with nh heads: the kernels
    index the [T, H, 128] rows, the per-head chunk tables and every
    workspace array by H, and the other tests use 8.  The saving pair on the
    same inputs must give the same bits."""
    from oracle import gated_delta, kimi_delta
    oracle_mod = kimi_delta if per_channel else gated_delta
    inp = synth.make_gdn_inputs(HEAD_CASE_CU, nh, 128, tensor_seed=11, per_channel=per_channel)
    scale = 1 / np.sqrt(128)
    if per_channel:
        from tests import test_kda as t
        tol_o, tol_g = t.TOL_O, {nm: t.TOL_GRAD for nm in ("dq", "dk", "dv", "dg", "dbeta")}
        run, run_bwd = t._run, t._run_bwd
    else:
        tol_o, tol_g, run, run_bwd = TOL_O, TOL_GRAD, _run, _run_bwd
    got = run(inp, scale).double().cpu().numpy()
    ref = oracle_mod.forward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens, scale)
    assert np.isfinite(got).all()
    assert rel_l2(got, ref) <= tol_o, rel_l2(got, ref)
    assert_per_segment(got, ref, inp.cu_seqlens, tol_o, "o")
    grads = run_bwd(inp, scale)
    refs = oracle_mod.backward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.do, inp.cu_seqlens, scale)
    for nm, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), grads, refs):
        assert np.isfinite(a).all(), nm
        assert rel_l2(a, b) <= tol_g[nm], (nm, rel_l2(a, b))
        assert_per_segment(a, b, inp.cu_seqlens, tol_g[nm], nm)
    # the saving pair on the same inputs: the same bits as the calls above
    import torch
    from varlen_sliding_window_gb300 import binding as b
    pre = "kda" if per_channel else "gdn"
    q, k, v, do = (_to_dev(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    g = torch.from_numpy(inp.g).cuda()
    beta = torch.from_numpy(inp.beta).cuda()
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    T = q.shape[0]
    ws = torch.empty(getattr(b, f"{pre}_varlen_bwd_workspace_bytes")(T, nh, len(inp.cu_seqlens) - 1),
                     dtype=torch.uint8, device="cuda")
    o2 = torch.empty_like(q)
    g2 = [torch.empty_like(q) for _ in range(3)] + [torch.empty_like(g), torch.empty_like(beta)]
    getattr(b, f"{pre}_varlen_fwd_save")(q, k, v, g, beta, cu, scale, o2, ws)
    getattr(b, f"{pre}_varlen_bwd_saved")(q, k, v, g, beta, do, cu, scale, *g2, ws)
    torch.cuda.synchronize()
    assert b.attn_varlen_get_status() == 0
    assert np.array_equal(o2.double().cpu().numpy(), got)
    for nm, a, c in zip(("dq", "dk", "dv", "dg", "dbeta"), grads, g2):
        assert np.array_equal(c.double().cpu().numpy(), a), nm


@pytest.mark.gpu
@pytest.mark.parametrize("nh", [1, 3, 5])
def test_head_counts(nh):
    check_head_counts(nh, per_channel=False)
