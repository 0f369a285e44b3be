"""Pins for the float64 oracle, independent of the oracle itself.

Each check is chosen so that a plausible mistake (a dropped term, a wrong sign
or index, a transposed operand, an off-by-one window, a leaking segment)
fails at least one of them: finite differences, closed forms, invariants,
hand-derived fixtures and torch's own float64 scaled_dot_product_attention.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from varlen_sliding_window_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, rng):
    return rng.standard_normal(shape)


def _small_case(rng, cu, hq=4, hkv=2, d=8):
    T = int(cu[-1])
    return (_rand((T, hq, d), rng), _rand((T, hkv, d), rng), _rand((T, hkv, d), rng), _rand((T, hq, d), rng))


def _parse(x):
    """Golden files spell ln-expressions as strings like 'ln3' or '-0.75ln3'."""
    if isinstance(x, list):
        return [_parse(y) for y in x]
    if isinstance(x, str):
        coef, _, arg = x.partition("ln")
        c = 1.0 if coef in ("", "+") else (-1.0 if coef == "-" else float(coef))
        return c * math.log(float(arg))
    return float(x)


@pytest.mark.parametrize("name", ["hand_two_token.json", "hand_window.json"])
def test_hand_derived_fixtures(name):
    g = json.load(open(os.path.join(GOLDEN, name)))
    q, k, v = (np.array(_parse(g[n])) for n in ("q", "k", "v"))
    out, lse = oracle.forward(q, k, v, g["cu_seqlens"], g["window_left"], g["softmax_scale"])
    np.testing.assert_allclose(out, np.array(_parse(g["out"])), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(_parse(g["lse"])), rtol=0, atol=1e-12)
    if "dq" in g:
        dout = np.array(_parse(g["dout"]))
        dq, dk, dv = oracle.backward(dout, q, k, v, g["cu_seqlens"], g["window_left"], g["softmax_scale"])
        np.testing.assert_allclose(dq, np.array(_parse(g["dq"])), atol=1e-12)
        np.testing.assert_allclose(dk, np.array(_parse(g["dk"])), atol=1e-12)
        np.testing.assert_allclose(dv, np.array(_parse(g["dv"])), atol=1e-12)


@pytest.mark.parametrize("window", [-1, 2])
def test_finite_differences(window):
    """Central differences of L = sum(dout * out) against the analytic backward."""
    rng = np.random.default_rng(7)
    cu = [0, 5, 14, 17]
    q, k, v, do = _small_case(rng, cu)
    scale = 0.4
    dq, dk, dv = oracle.backward(do, q, k, v, cu, window, scale)

    def loss(qq, kk, vv):
        return float((oracle.forward(qq, kk, vv, cu, window, scale)[0] * do).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.linalg.norm(num - g) / np.linalg.norm(g)
        assert err < 1e-7, (name, err)


def test_rows_of_p_sum_to_one():
    rng = np.random.default_rng(1)
    cu = [0, 37, 100]
    q, k, v, _ = _small_case(rng, cu, d=16)
    for window in (-1, 0, 5):
        for s in range(2):
            for h in range(4):
                p = oracle.probabilities(q, k, cu, window, 0.3, s, h)
                np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
                # Nothing above the diagonal, nothing outside the window.
                assert np.all(np.triu(p, 1) == 0)
                if window >= 0:
                    assert np.all(np.tril(p, -window - 1) == 0)


def test_large_window_equals_global():
    rng = np.random.default_rng(2)
    cu = [0, 20, 33, 64]
    q, k, v, do = _small_case(rng, cu)
    ref = oracle.forward(q, k, v, cu, -1, 0.35)
    got = oracle.forward(q, k, v, cu, 19, 0.35)  # longest segment is 31 -> 19 < 30 differs
    assert not np.array_equal(ref[0], got[0])
    got = oracle.forward(q, k, v, cu, 30, 0.35)
    assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[1], got[1])
    gref = oracle.backward(do, q, k, v, cu, -1, 0.35)
    gwin = oracle.backward(do, q, k, v, cu, 1000, 0.35)
    for a, b in zip(gref, gwin):
        assert np.array_equal(a, b)


def test_segment_isolation():
    """Perturbing one document leaves every other one bit-identical."""
    rng = np.random.default_rng(3)
    cu = [0, 9, 30, 31, 50]
    q, k, v, do = _small_case(rng, cu)
    for window in (-1, 4):
        base = oracle.forward(q, k, v, cu, window, 0.3) + oracle.backward(do, q, k, v, cu, window, 0.3)
        q2, k2, v2, do2 = q.copy(), k.copy(), v.copy(), do.copy()
        sl = slice(9, 30)
        for t in (q2, k2, v2, do2):
            t[sl] += rng.standard_normal(t[sl].shape)
        pert = oracle.forward(q2, k2, v2, cu, window, 0.3) + oracle.backward(do2, q2, k2, v2, cu, window, 0.3)
        out, lse, dq, dk, dv = base
        out2, lse2, dq2, dk2, dv2 = pert
        outside = np.r_[0:9, 30:50]
        assert np.array_equal(out[outside], out2[outside])
        assert np.array_equal(lse[:, outside], lse2[:, outside])
        for a, b in ((dq, dq2), (dk, dk2), (dv, dv2)):
            assert np.array_equal(a[outside], b[outside])
        assert not np.allclose(out[sl], out2[sl])


def test_gqa_equals_mha_with_repeated_kv():
    rng = np.random.default_rng(4)
    cu = [0, 12, 40]
    hq, hkv = 8, 2
    q, k, v, do = _small_case(rng, cu, hq=hq, hkv=hkv)
    rep = hq // hkv
    kr, vr = np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1)
    for window in (-1, 3):
        o1, l1 = oracle.forward(q, k, v, cu, window, 0.3)
        o2, l2 = oracle.forward(q, kr, vr, cu, window, 0.3)
        np.testing.assert_allclose(o1, o2, atol=1e-13)
        np.testing.assert_allclose(l1, l2, atol=1e-13)
        g1 = oracle.backward(do, q, k, v, cu, window, 0.3)
        g2 = oracle.backward(do, q, kr, vr, cu, window, 0.3)
        np.testing.assert_allclose(g1[0], g2[0], atol=1e-12)
        np.testing.assert_allclose(g1[1], g2[1].reshape(-1, hkv, rep, 8).sum(axis=2), atol=1e-12)
        np.testing.assert_allclose(g1[2], g2[2].reshape(-1, hkv, rep, 8).sum(axis=2), atol=1e-12)


def test_closed_forms():
    rng = np.random.default_rng(5)
    # Length-1 segments: out = v, lse = scale <q, k>.
    cu = list(range(0, 7))
    q, k, v, _ = _small_case(rng, cu)
    out, lse = oracle.forward(q, k, v, cu, -1, 0.7)
    g = np.arange(4) // 2
    np.testing.assert_allclose(out, v[:, g], atol=1e-14)
    np.testing.assert_allclose(lse, 0.7 * np.einsum("thd,thd->ht", q, k[:, g]), atol=1e-13)
    # window 0: every query sees only itself.
    cu = [0, 11, 25]
    q, k, v, _ = _small_case(rng, cu)
    out, _ = oracle.forward(q, k, v, cu, 0, 0.7)
    np.testing.assert_allclose(out, v[:, g], atol=1e-14)
    # q == 0: uniform weights, out = mean of visible v, lse = ln |V(i)|.
    for window in (-1, 3):
        out, lse = oracle.forward(np.zeros_like(q), k, v, cu, window, 0.7)
        for a, b in ((0, 11), (11, 25)):
            for i in range(a, b):
                lo = a if window < 0 else max(a, i - window)
                np.testing.assert_allclose(out[i], v[lo:i + 1][:, g].mean(axis=0), atol=1e-14)
                np.testing.assert_allclose(lse[:, i], math.log(i + 1 - lo), atol=1e-14)


def test_gradient_sum_invariants():
    """Per segment and kv head: sum_j dk = 0 and sum_j dv = sum over group of sum_i dout."""
    rng = np.random.default_rng(6)
    cu = [0, 13, 31, 32, 60]
    q, k, v, do = _small_case(rng, cu)
    for window in (-1, 2):
        dq, dk, dv = oracle.backward(do, q, k, v, cu, window, 0.3)
        for a, b in oracle.segments(cu):
            np.testing.assert_allclose(dk[a:b].sum(axis=0), 0.0, atol=1e-12)
            dsum = do[a:b].reshape(b - a, 2, 2, 8).sum(axis=(0, 2))
            np.testing.assert_allclose(dv[a:b].sum(axis=0), dsum, atol=1e-12)


def test_empty_segments_change_nothing():
    rng = np.random.default_rng(8)
    cu = np.array([0, 10, 21, 40])
    q, k, v, do = _small_case(rng, cu)
    padded = np.array([0, 0, 10, 10, 21, 40, 40, 40])
    for window in (-1, 3):
        a = oracle.forward(q, k, v, cu, window, 0.3) + oracle.backward(do, q, k, v, cu, window, 0.3)
        b = oracle.forward(q, k, v, padded, window, 0.3) + oracle.backward(do, q, k, v, padded, window, 0.3)
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


@pytest.mark.parametrize("window", [-1, 6])
def test_matches_torch_sdpa_float64(window):
    """torch's float64 SDPA (a different library, with its own mask handling)
    and torch autograd agree with the oracle's forward and analytic backward."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(9)
    cu = [0, 17, 40, 41, 64]
    hq, hkv, d = 4, 2, 16
    q, k, v, do = _small_case(rng, cu, hq=hq, hkv=hkv, d=d)
    scale = 0.25
    T = cu[-1]
    seg = np.zeros(T, dtype=np.int64)
    for s, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        seg[a:b] = s
    tseg = torch.from_numpy(seg)
    pos = torch.arange(T)
    allowed = (tseg[:, None] == tseg[None, :]) & (pos[None, :] <= pos[:, None])
    if window >= 0:
        allowed &= (pos[:, None] - pos[None, :]) <= window
    tq = torch.from_numpy(q).permute(1, 0, 2).requires_grad_(True)  # [H, T, d]
    tk = torch.from_numpy(k).repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2).detach().requires_grad_(True)
    tv = torch.from_numpy(v).repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2).detach().requires_grad_(True)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=allowed, scale=scale)
    o.backward(torch.from_numpy(do).permute(1, 0, 2))
    out, _ = oracle.forward(q, k, v, cu, window, scale)
    dq, dk, dv = oracle.backward(do, q, k, v, cu, window, scale)
    np.testing.assert_allclose(out, o.detach().permute(1, 0, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.permute(1, 0, 2).numpy(), atol=1e-11)
    tdk = tk.grad.permute(1, 0, 2).numpy().reshape(T, hkv, hq // hkv, d).sum(axis=2)
    tdv = tv.grad.permute(1, 0, 2).numpy().reshape(T, hkv, hq // hkv, d).sum(axis=2)
    np.testing.assert_allclose(dk, tdk, atol=1e-11)
    np.testing.assert_allclose(dv, tdv, atol=1e-11)


def test_single_segment_is_torch_causal():
    """A single global-causal segment is exactly SDPA(is_causal=True)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(10)
    q, k, v, _ = _small_case(rng, [0, 50], hq=2, hkv=2, d=32)
    o = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).permute(1, 0, 2), torch.from_numpy(k).permute(1, 0, 2),
        torch.from_numpy(v).permute(1, 0, 2), is_causal=True, scale=0.2)
    out, _ = oracle.forward(q, k, v, [0, 50], -1, 0.2)
    np.testing.assert_allclose(out, o.permute(1, 0, 2).numpy(), atol=1e-12)


def test_row_blocking_is_invisible(monkeypatch):
    """Cutting long segments into blocks of query rows changes nothing."""
    import oracle.attention as oa
    rng = np.random.default_rng(11)
    cu = [0, 70, 75]
    q, k, v, do = _small_case(rng, cu)
    a = oa.forward(q, k, v, cu, -1, 0.3) + oa.backward(do, q, k, v, cu, -1, 0.3)
    monkeypatch.setattr(oa, "ROW_BLOCK", 16)
    b = oa.forward(q, k, v, cu, -1, 0.3) + oa.backward(do, q, k, v, cu, -1, 0.3)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-12)


def test_visible_ranges_and_pair_counts():
    cu = [0, 61, 161, 256]
    for window in (-1, 64):
        r = oracle.visible_ranges(cu, window, 256)
        assert r[:, 2].sum() == oracle.unmasked_pairs(cu, window)
        for a, b in ((0, 61), (61, 161), (161, 256)):
            L = b - a
            i = np.arange(a, b)
            if window < 0:
                assert r[a:b, 2].sum() == L * (L + 1) // 2
                first = np.full(L, a)
            else:
                # The window reaches back w keys but never past the segment start.
                first = np.maximum(a, i - window)
            np.testing.assert_array_equal(r[a:b, 0], first)
            np.testing.assert_array_equal(r[a:b, 1], i)
            np.testing.assert_array_equal(r[a:b, 2], i - first + 1)
    # Closed form for the 3-document workload: 61*62/2 + 100*101/2 + 95*96/2.
    assert oracle.unmasked_pairs(cu, -1) == 1891 + 5050 + 4560


def test_generator_matches_page_statistics():
    """Document lengths: median 457 and ~45 % of tokens in documents >= 4,096
    (research.dws.rip/llm/kernels, section 01)."""
    lengths = np.array(synth.draw_document_lengths(3_000_000, 123))
    assert abs(np.median(lengths) / 457.0 - 1) < 0.03
    share = lengths[lengths >= 4096].sum() / lengths.sum()
    assert 0.40 < share < 0.50
    cu = synth.pack_microbatch(16384, 4096, 0)
    assert cu[0] == 0 and cu[-1] == 16384 and np.all(np.diff(cu) > 0)
    assert np.all(np.diff(cu) <= 4096)
    assert set(range(0, 16385, 4096)) <= set(cu.tolist())


def test_bf16_rounding():
    bits, vals = synth.round_to_bf16(np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e-3], dtype=np.float32))
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: rounds to even (1.0).
    assert vals[0] == 1.0 and vals[1] == 1.0 and vals[2] == np.float32(1.0078125)
    assert vals[3] == -2.5 and bits[0] == 0x3F80
