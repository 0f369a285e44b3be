"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (relative L2, over the whole tensor and again over every segment on
its own): out <= 5e-3, dq/dk/dv <= 1e-2; lse within 1e-3 absolute.  Which keys
each query sees is checked bit-exactly.
"""
import numpy as np
import pytest

import oracle
from varlen_sliding_window_gb300 import synth

from helpers import (TOL_GRAD, TOL_LSE_ABS, TOL_OUT, assert_per_segment, by_key_ranges_from_oracle, rel_l2,
                     run_gpu, segment_slice, to_device_bf16)

pytestmark = pytest.mark.gpu

WL = synth.workloads()


def _check_full(inp, window, scale, max_seqlen, res):
    ref_out, ref_lse = oracle.forward(inp.q, inp.k, inp.v, inp.cu_seqlens, window, scale)
    dq, dk, dv = oracle.backward(inp.dout, inp.q, inp.k, inp.v, inp.cu_seqlens, window, scale)
    errs = {"out": rel_l2(res["out"], ref_out)}
    assert errs["out"] <= TOL_OUT, errs
    for g, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
        if np.linalg.norm(ref) < 1e-9:
            # window_left = 0: every query sees only itself, P = 1 and
            # dS = dP - D = 0, so dq and dk vanish exactly; the GPU's D comes
            # from the bf16-rounded out, leaving rounding-level residue.
            errs[g] = float(np.sqrt(np.mean(res[g] ** 2)))
            assert errs[g] <= 1e-4, errs
        else:
            errs[g] = rel_l2(res[g], ref)
            assert errs[g] <= TOL_GRAD, errs
    assert np.abs(res["lse"] - ref_lse).max() <= TOL_LSE_ABS
    cu = inp.cu_seqlens
    errs["out_seg"] = assert_per_segment(res["out"], ref_out, cu, TOL_OUT, "out")
    for g, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
        errs[g + "_seg"] = assert_per_segment(res[g], ref, cu, TOL_GRAD, g)
    return errs


@pytest.mark.parametrize("name", ["tiny_global", "tiny_w64"])
def test_tiny_workloads(name):
    wl = WL[name]
    inp = wl.inputs()
    res = run_gpu(inp, wl.window_left, wl.softmax_scale, 256)
    _check_full(inp, wl.window_left, wl.softmax_scale, 256, res)


@pytest.mark.parametrize("window", [-1, 0, 1, 64, 127, 128, 129, 300, 512])
def test_ragged_multi_tile(window):
    """Segments spanning several tiles with ragged tails, a length-1 segment,
    an exact tile multiple, and both global and many window widths."""
    cu = np.array([0, 1, 130, 386, 387, 900, 1024, 1536, 1800], dtype=np.int32)
    inp = synth.make_inputs(cu, 8, 2, 128, tensor_seed=3)
    res = run_gpu(inp, window, 1 / np.sqrt(128), 600)
    _check_full(inp, window, 1 / np.sqrt(128), 600, res)


@pytest.mark.parametrize("window", [4095, 4096, 4097])
def test_very_large_window(window):
    """Windows of about 4,096 tokens (the packed sliding-window benchmark of
    dewml.dev/reference/performance) on segments longer than the window:
    each 128-query tile sees the kv tiles of its band, [i - w, i], up to 33
    of them; compared in full with the oracle, per segment too."""
    cu = np.array([0, 5000, 5001, 9100, 9500], dtype=np.int32)
    inp = synth.make_inputs(cu, 8, 2, 128, tensor_seed=8)
    res = run_gpu(inp, window, 1 / np.sqrt(128), 5000)
    _check_full(inp, window, 1 / np.sqrt(128), 5000, res)


@pytest.mark.parametrize("hq,hkv", [(8, 2), (16, 4), (4, 4), (6, 2), (8, 1)])
def test_head_ratios(hq, hkv):
    cu = np.array([0, 200, 333, 700], dtype=np.int32)
    inp = synth.make_inputs(cu, hq, hkv, 128, tensor_seed=4)
    for window in (-1, 100):
        res = run_gpu(inp, window, 0.0884, 400)
        _check_full(inp, window, 0.0884, 400, res)


@pytest.mark.parametrize("window", [-1, 2])
def test_many_tiny_segments(window):
    """8,000 segments of 1 to 4 tokens (about 20,000 tokens): more work tiles
    than the all-thread planner holds, so every kernel takes its single-warp
    fallback scheduler, and more work units than one persistent CTA per SM
    can own, so the grids grow past the SM count.  Compared in full."""
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 5, size=8000)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    inp = synth.make_inputs(cu, 8, 2, 128, tensor_seed=21)
    res = run_gpu(inp, window, 1 / np.sqrt(128), 4)
    _check_full(inp, window, 1 / np.sqrt(128), 4, res)


def _group_slice(inp, a: int, b: int, g: int, hq: int, hkv: int):
    """Segment [a, b) restricted to kv head g and its query heads, as a
    standalone one-segment problem with Hq/Hkv query heads and one kv head."""
    import copy
    grp = hq // hkv
    sub = copy.copy(inp)
    sub.q = inp.q[a:b, g * grp:(g + 1) * grp]
    sub.dout = inp.dout[a:b, g * grp:(g + 1) * grp]
    sub.k = inp.k[a:b, g:g + 1]
    sub.v = inp.v[a:b, g:g + 1]
    sub.cu_seqlens = np.array([0, b - a], dtype=np.int32)
    return sub


@pytest.mark.parametrize("name", ["ctx512_global", "ctx4096_w512", "ctx4096_global", "long65536_global",
                                  "long65536_w4096"])
def test_full_size_sampled_segments(name):
    """At the full sizes (the benchmark's launch configuration for the
    16,384-token microbatches; 65,536 tokens with 16/4 heads for the long
    case), the oracle is run on a sample of whole segments (first, last,
    longest, shortest, and one in the middle), each compared on its own;
    every segment is independent.  In the long case the sample is taken
    among segments of at most 2,048 tokens with all 16 heads, and the two
    longest segments (several thousand tokens: the dK/dV pass splits their
    kv tiles into the longest chains) are compared on one kv group (query
    heads 0-3 and kv head 0), which keeps the float64 oracle within tens of
    seconds."""
    wl = WL[name]
    inp = wl.inputs()
    res = run_gpu(inp, wl.window_left, wl.softmax_scale, wl.context)
    cu = inp.cu_seqlens
    lens = np.diff(cu)
    cap = 2048 if wl.total > 16384 else wl.total
    longest = int(np.argmax(np.where(lens <= cap, lens, -1)))
    picks = sorted({0, len(lens) - 1, longest, int(np.argmin(lens)), len(lens) // 2})
    picks = [s for s in picks if lens[s] <= cap] or [int(np.argmin(lens))]
    for s in picks:
        a, b = int(cu[s]), int(cu[s + 1])
        sub = segment_slice(inp, a, b)
        ref_out, ref_lse = oracle.forward(sub.q, sub.k, sub.v, sub.cu_seqlens, wl.window_left, wl.softmax_scale)
        g = oracle.backward(sub.dout, sub.q, sub.k, sub.v, sub.cu_seqlens, wl.window_left, wl.softmax_scale)
        assert rel_l2(res["out"][a:b], ref_out) <= TOL_OUT, (s, "out")
        assert np.abs(res["lse"][:, a:b] - ref_lse).max() <= TOL_LSE_ABS
        for nm, got, ref in zip(("dq", "dk", "dv"), (res["dq"][a:b], res["dk"][a:b], res["dv"][a:b]), g):
            assert rel_l2(got, ref) <= TOL_GRAD, (s, nm)
    if wl.total > 16384:
        grp = wl.hq // wl.hkv
        for s in np.argsort(lens)[::-1][:2]:
            a, b = int(cu[s]), int(cu[s + 1])
            assert b - a > cap  # these segments are outside the all-head sample
            sub = _group_slice(inp, a, b, 0, wl.hq, wl.hkv)
            ref_out, ref_lse = oracle.forward(sub.q, sub.k, sub.v, sub.cu_seqlens, wl.window_left, wl.softmax_scale)
            g = oracle.backward(sub.dout, sub.q, sub.k, sub.v, sub.cu_seqlens, wl.window_left, wl.softmax_scale)
            assert rel_l2(res["out"][a:b, :grp], ref_out) <= TOL_OUT, (s, "out")
            assert np.abs(res["lse"][:grp, a:b] - ref_lse).max() <= TOL_LSE_ABS
            got = (res["dq"][a:b, :grp], res["dk"][a:b, :1], res["dv"][a:b, :1])
            for nm, x, ref in zip(("dq", "dk", "dv"), got, g):
                assert rel_l2(x, ref) <= TOL_GRAD, (s, nm)
    # Properties that hold for every segment at any size.
    assert np.all(np.isfinite(res["out"])) and np.all(np.isfinite(res["dq"]))
    # Per segment, kv head and column: sum_j dk = 0 and sum_j dv = sum of dout
    # over the group.  The GPU values carry bf16 rounding (2^-9 relative) and
    # the kernel's own error (~3e-3 of the column norm), which add up like a
    # random walk over the rows, so the bound is 3 % of the column's L2 norm.
    for a, b in oracle.segments(cu):
        dk = res["dk"][a:b]
        assert np.all(np.abs(dk.sum(axis=0)) <= 3e-2 * np.linalg.norm(dk, axis=0) + 1e-3)
        dv = res["dv"][a:b]
        do_sum = inp.dout[a:b].astype(np.float64).reshape(b - a, wl.hkv, wl.hq // wl.hkv, 128).sum(axis=(0, 2))
        assert np.all(np.abs(dv.sum(axis=0) - do_sum) <= 3e-2 * np.linalg.norm(dv, axis=0) + 1e-2)


def _padded(cu: np.ndarray) -> np.ndarray:
    """cu_seqlens with empty segments at the front, in the middle and at the end."""
    m = len(cu) // 2
    return np.concatenate([[0, 0, 0], cu[1:m], [cu[m - 1]] * 2, cu[m:], [cu[-1]] * 5]).astype(np.int32)


def _cu_of(name: str) -> tuple:
    """(workload, cu_seqlens) for a workload name, '+pad' = padded with empty segments."""
    base = name.removesuffix("+pad")
    wl = WL[base]
    cu = wl.cu_seqlens()
    return wl, (_padded(cu) if name.endswith("+pad") else cu)


MASK_CASES = ["tiny_global", "tiny_w64", "tiny_w64+pad", "ctx512_global", "ctx4096_w512", "ctx4096_w512+pad",
              "ctx4096_global", "ctx4096_global+pad", "long65536_global", "long65536_w4096"]


@pytest.mark.parametrize("name", MASK_CASES)
def test_mask_ranges_bit_exact(name):
    """The kernels' own mask/tile logic, exported by the test hook, against the
    oracle's visible sets, per query and per key (plain and padded boundary
    lists)."""
    import torch
    from varlen_sliding_window_gb300 import binding
    wl, cu = _cu_of(name)
    T = int(cu[-1])
    dcu = torch.from_numpy(cu).cuda()
    ranges = torch.empty(3 * T, dtype=torch.int32, device="cuda")
    binding.attn_varlen_mask_ranges(dcu, T, wl.context, wl.window_left, False, ranges)
    got = ranges.view(T, 3).cpu().numpy().astype(np.int64)
    np.testing.assert_array_equal(got, oracle.visible_ranges(cu, wl.window_left, T))
    binding.attn_varlen_mask_ranges(dcu, T, wl.context, wl.window_left, True, ranges)
    got = ranges.view(T, 3).cpu().numpy().astype(np.int64)
    np.testing.assert_array_equal(got, by_key_ranges_from_oracle(cu, wl.window_left, T))


@pytest.mark.parametrize("name", MASK_CASES)
def test_zero_q_counts_visible_keys(name):
    """With q = 0 every visible key has the same logit, so exp(lse) is exactly
    the number of keys the real forward kernel let each query see (plain and
    padded boundary lists)."""
    wl, cu = _cu_of(name)
    inp = synth.make_inputs(cu, wl.hq, wl.hkv, wl.d, wl.tensor_seed)
    inp.q_bits = np.zeros_like(inp.q_bits)
    res = run_gpu(inp, wl.window_left, wl.softmax_scale, wl.context, backward=False)
    counts = oracle.visible_ranges(cu, wl.window_left, wl.total)[:, 2]
    np.testing.assert_array_equal(np.rint(np.exp(res["lse"])).astype(np.int64), np.broadcast_to(counts, res["lse"].shape))


def test_empty_segments_are_bit_identical():
    """Padding cu_seqlens with empty segments (front, middle, end) changes no bit."""
    wl = WL["ctx4096_w512"]
    inp = wl.inputs()
    cu = inp.cu_seqlens
    padded = np.concatenate([[0, 0], cu[1:5], [cu[4]] * 3, cu[5:], [cu[-1]] * 4]).astype(np.int32)
    a = run_gpu(inp, wl.window_left, wl.softmax_scale, wl.context)
    b = run_gpu(inp, wl.window_left, wl.softmax_scale, wl.context, cu_override=padded)
    for key in ("out", "lse", "dq", "dk", "dv"):
        assert np.array_equal(a[key], b[key]), key


def test_deterministic():
    wl = WL["ctx4096_global"]
    inp = wl.inputs()
    a = run_gpu(inp, wl.window_left, wl.softmax_scale, wl.context)
    b = run_gpu(inp, wl.window_left, wl.softmax_scale, wl.context)
    for key in ("out", "lse", "dq", "dk", "dv"):
        assert np.array_equal(a[key], b[key]), key


@pytest.mark.parametrize("window", [-1, 512])
def test_repeated_backward_is_bitwise_stable(window):
    """The backward run many times on the same device-resident inputs gives
    the same bits every time and no non-finite value.  Warp timing differs
    from run to run, so this catches barrier races that only show
    occasionally (a warp lapping its warpgroup, a buffer reused too early)."""
    import torch
    from varlen_sliding_window_gb300 import binding
    cu = synth.pad_cu_seqlens(synth.pack_microbatch(16384, 4096, 3), 48)
    inp = synth.make_inputs(cu, 8, 2, 128, tensor_seed=13)
    q, k, v, do = (to_device_bf16(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits, inp.dout_bits))
    cu_d = torch.from_numpy(np.asarray(cu, dtype=np.int32)).cuda()
    out = torch.empty_like(q)
    lse = torch.empty(8, q.shape[0], dtype=torch.float32, device="cuda")
    scale = 128 ** -0.5
    binding.attn_varlen_get_status()  # start from a clear status word
    binding.attn_varlen_fwd(q, k, v, cu_d, 4096, window, scale, out, lse)
    ref = None
    for _ in range(10):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        binding.attn_varlen_bwd(do, q, k, v, out, lse, cu_d, 4096, window, scale, dq, dk, dv)
        torch.cuda.synchronize()
        got = (dq, dk, dv)
        for t in got:
            assert torch.isfinite(t.float()).all()
        if ref is None:
            ref = tuple(t.clone() for t in got)
        else:
            for name, a, b in zip(("dq", "dk", "dv"), ref, got):
                assert torch.equal(a, b), name
    assert binding.attn_varlen_get_status() == 0


@pytest.mark.parametrize("window", [-1, 512])
def test_cuda_graph_replay_matches_eager(window):
    """Forward + backward captured once in a CUDA graph with the boundary list
    padded to 42 segments (research.dws.rip/llm/kernels, section 06 and
    Fig. 8), replayed over three batches with different boundaries: each replay
    matches eager runs bit for bit, both on the same padded list and on the
    unpadded one."""
    import torch
    from varlen_sliding_window_gb300 import binding
    wl = WL["ctx4096_w512"]
    nseg_pad = 42
    batches = []
    for seed in (0, 1, 2):
        cu = synth.pack_microbatch(16384, 4096, seed)
        assert len(cu) - 1 <= nseg_pad
        batches.append((cu, synth.pad_cu_seqlens(cu, nseg_pad), synth.make_inputs(cu, 8, 2, 128, tensor_seed=10 + seed)))
    assert len({len(c) for c, _, _ in batches}) > 1  # the batches differ in their segment counts
    dev = torch.device("cuda")
    q = torch.empty(16384, 8, 128, dtype=torch.bfloat16, device=dev)
    k = torch.empty(16384, 2, 128, dtype=torch.bfloat16, device=dev)
    v, do = torch.empty_like(k), torch.empty_like(q)
    cu_d = torch.zeros(nseg_pad + 1, dtype=torch.int32, device=dev)
    out, dq = torch.empty_like(q), torch.empty_like(q)
    dk, dv = torch.empty_like(k), torch.empty_like(k)
    lse = torch.empty(8, 16384, dtype=torch.float32, device=dev)
    outs = (out, lse, dq, dk, dv)

    def load(cu_pad, inp):
        cu_d.copy_(torch.from_numpy(cu_pad))
        for dst, bits in ((q, inp.q_bits), (k, inp.k_bits), (v, inp.v_bits), (do, inp.dout_bits)):
            dst.copy_(to_device_bf16(bits))

    def step(cu):
        binding.attn_varlen_fwd(q, k, v, cu, 4096, window, wl.softmax_scale, out, lse)
        binding.attn_varlen_bwd(do, q, k, v, out, lse, cu, 4096, window, wl.softmax_scale, dq, dk, dv)

    s = torch.cuda.Stream()
    load(*batches[0][1:])
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step(cu_d)  # warm-up (allocator pool, function attributes) outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(cu_d)
    for cu, cu_pad, inp in batches:
        load(cu_pad, inp)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        replayed = [t.clone() for t in outs]
        for t in outs:
            t.fill_(float("nan"))
        step(cu_d)
        torch.cuda.synchronize()
        for x, y in zip(replayed, outs):
            assert torch.equal(x, y)
        for t in outs:
            t.fill_(float("nan"))
        step(torch.from_numpy(cu).to(dev))
        torch.cuda.synchronize()
        for x, y in zip(replayed, outs):
            assert torch.equal(x, y)
    assert binding.attn_varlen_get_status() == 0
