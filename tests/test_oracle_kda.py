"""Pins for the Kimi Delta oracle, independent of the oracle itself.

Finite differences of every input, torch float64 autograd through the
paper's form of the step, Gated DeltaNet (its own pins in
test_oracle_gdn.py) when the gate is equal on every channel, closed forms,
segment isolation, empty segments, and a chunked evaluation written here from
the algebra.
"""
import numpy as np
import pytest

from oracle import gated_delta as gdn
from oracle import kimi_delta as kda


def _case(rng, cu, nh=2, dk=3, dv=4, gate_scale=1.0):
    T = int(cu[-1])
    q = rng.standard_normal((T, nh, dk)) / np.sqrt(dk)
    k = rng.standard_normal((T, nh, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, nh, dv))
    g = -gate_scale * np.log1p(np.exp(rng.standard_normal((T, nh, dk))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, nh))))
    do = rng.standard_normal((T, nh, dv))
    return q, k, v, g, beta, do


CU = np.array([0, 4, 4, 9], dtype=np.int32)


def test_finite_differences_every_input():
    rng = np.random.default_rng(0)
    q, k, v, g, beta, do = _case(rng, CU)
    scale = 0.6
    grads = kda.backward(q, k, v, g, beta, do, CU, scale)
    args = [q, k, v, g, beta]
    h = 1e-6
    for idx, (x, gx) in enumerate(zip(args, grads)):
        num = np.zeros_like(x)
        for pos in np.ndindex(x.shape):
            saved = x[pos]
            x[pos] = saved + h
            lp = np.sum(do * kda.forward(*args, CU, scale))
            x[pos] = saved - h
            lm = np.sum(do * kda.forward(*args, CU, scale))
            x[pos] = saved
            num[pos] = (lp - lm) / (2 * h)
        err = np.max(np.abs(num - gx)) / max(np.max(np.abs(num)), 1e-12)
        assert err < 1e-7, (idx, err)


def test_torch_autograd_through_the_papers_step():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    cu = np.array([0, 7, 7, 15], dtype=np.int32)
    q, k, v, g, beta, do = _case(rng, cu, nh=2, dk=5, dv=3)
    scale = 0.5
    ts = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v, g, beta)]
    tq, tk, tv, tg, tb = ts
    outs = []
    eye = torch.eye(5, dtype=torch.float64)
    for a, b in zip(cu[:-1], cu[1:]):
        S = torch.zeros(2, 5, 3, dtype=torch.float64)  # [H, dk, dv]
        for t in range(int(a), int(b)):
            kk = tk[t][:, :, None] * tk[t][:, None, :]
            S = (eye - tb[t][:, None, None] * kk) @ (torch.exp(tg[t])[:, :, None] * S) + tb[t][:, None, None] * (
                tk[t][:, :, None] * tv[t][:, None, :])
            outs.append(scale * torch.einsum("hkv,hk->hv", S, tq[t]))
    o = torch.stack(outs)
    np.testing.assert_allclose(o.detach().numpy(), kda.forward(q, k, v, g, beta, cu, scale), rtol=1e-12, atol=1e-12)
    (o * torch.tensor(do)).sum().backward()
    for t, mine in zip(ts, kda.backward(q, k, v, g, beta, do, cu, scale)):
        np.testing.assert_allclose(mine, t.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_equal_channels_is_gated_deltanet():
    rng = np.random.default_rng(2)
    cu = np.array([0, 6, 13], dtype=np.int32)
    q, k, v, g, beta, do = _case(rng, cu, dk=4)
    g1 = g[:, :, 0]
    gk = np.repeat(g1[:, :, None], 4, axis=2)
    np.testing.assert_allclose(kda.forward(q, k, v, gk, beta, cu), gdn.forward(q, k, v, g1, beta, cu),
                               rtol=1e-13, atol=1e-14)
    a = kda.backward(q, k, v, gk, beta, do, cu)
    b = gdn.backward(q, k, v, g1, beta, do, cu)
    for i in (0, 1, 2, 4):
        np.testing.assert_allclose(a[i], b[i], rtol=1e-12, atol=1e-13)
    # the scalar gate's gradient is the sum of the channel gates' gradients
    np.testing.assert_allclose(a[3].sum(axis=2), b[3], rtol=1e-12, atol=1e-13)


def test_single_write_decays_per_channel():
    # beta = 1 at the first token, 0 afterwards: S_t = Diag(prod_{j=1..t} alpha_j) k_0 v_0^T.
    rng = np.random.default_rng(3)
    cu = np.array([0, 6], dtype=np.int32)
    q, k, v, g, beta, _ = _case(rng, cu, dk=4)
    beta[:] = 0.0
    beta[0] = 1.0
    o = kda.forward(q, k, v, g, beta, cu, 1.0)
    for t in range(6):
        decay = np.exp(np.sum(g[1:t + 1], axis=0))  # [H, dk]
        want = np.sum(q[t] * decay * k[0], axis=-1)[:, None] * v[0]
        np.testing.assert_allclose(o[t], want, rtol=1e-12, atol=1e-14)


def test_zero_decay_keeps_only_the_current_token():
    rng = np.random.default_rng(4)
    q, k, v, g, beta, _ = _case(rng, CU)
    g[:] = -np.inf
    o = kda.forward(q, k, v, g, beta, CU, 0.9)
    want = 0.9 * beta[:, :, None] * np.sum(q * k, axis=-1)[:, :, None] * v
    np.testing.assert_allclose(o, want, rtol=1e-13, atol=1e-14)


def test_segments_are_isolated_and_empty_segments_change_nothing():
    rng = np.random.default_rng(5)
    cu = np.array([0, 5, 12, 20], dtype=np.int32)
    q, k, v, g, beta, do = _case(rng, cu)
    o = kda.forward(q, k, v, g, beta, cu)
    for a, b in zip(cu[:-1], cu[1:]):
        sub = [x[a:b] for x in (q, k, v, g, beta)]
        np.testing.assert_array_equal(kda.forward(*sub, np.array([0, b - a], np.int32)), o[a:b])
    cu_pad = np.array([0, 0, 5, 5, 12, 20, 20], dtype=np.int32)
    np.testing.assert_array_equal(kda.forward(q, k, v, g, beta, cu_pad), o)
    for x, y in zip(kda.backward(q, k, v, g, beta, do, cu_pad), kda.backward(q, k, v, g, beta, do, cu)):
        np.testing.assert_array_equal(x, y)


def _chunked(q, k, v, g, beta, cu, scale, C):
    """The chunked form, from the algebra: with gamma the running sum of g over
    the chunk (per channel) and B = exp(gamma),
    A_ij = beta_i <k_i o B_i, k_j / B_j> (j < i), X = (I + A)^-1,
    W = X diag(beta) (K o B), U = X diag(beta) V, E = U - W S0,
    O = scale ((Q o B) S0 + lower(<q_i o B_i, k_j / B_j>) E),
    S1 = Diag(B_last) S0 + (K o B_last / B)^T E."""
    T, nh, dk = k.shape
    o = np.zeros((T, nh, v.shape[2]))
    for a, b in zip(cu[:-1], cu[1:]):
        for h in range(nh):
            S0 = np.zeros((dk, v.shape[2]))
            for c0 in range(int(a), int(b), C):
                c1 = min(int(b), c0 + C)
                K, V, Q = k[c0:c1, h], v[c0:c1, h], q[c0:c1, h]
                B = np.exp(np.cumsum(g[c0:c1, h], axis=0))
                bt = beta[c0:c1, h]
                n = c1 - c0
                A = np.tril(bt[:, None] * ((K * B) @ (K / B).T), -1)
                X = np.linalg.inv(np.eye(n) + A)
                W = X @ (bt[:, None] * (K * B))
                U = X @ (bt[:, None] * V)
                E = U - W @ S0
                o[c0:c1, h] = scale * ((Q * B) @ S0 + np.tril((Q * B) @ (K / B).T) @ E)
                S0 = B[-1][:, None] * S0 + (K * (B[-1] / B)).T @ E
    return o


@pytest.mark.parametrize("C", [1, 3, 8])
def test_chunked_form_matches_the_recurrence(C):
    rng = np.random.default_rng(6)
    cu = np.array([0, 11, 11, 30, 33], dtype=np.int32)
    q, k, v, g, beta, _ = _case(rng, cu, nh=2, dk=6, dv=5, gate_scale=0.3)
    want = kda.forward(q, k, v, g, beta, cu, 0.4)
    np.testing.assert_allclose(_chunked(q, k, v, g, beta, cu, 0.4, C), want, rtol=1e-9, atol=1e-11)
