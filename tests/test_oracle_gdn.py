"""Pins for the Gated DeltaNet oracle, independent of the oracle itself.

Each check is chosen so that a plausible mistake (the gate applied after the
write instead of before it, beta on the wrong term, a transposed state, a
state leaking across a document boundary, a wrong sign in the backward)
fails at least one of them: central finite differences, torch float64
autograd through the recurrence, closed forms, invariants and a chunked
(WY-form) evaluation written here from the algebra, not from the oracle.
"""
import numpy as np
import pytest

from oracle import gated_delta as gdn


def _case(rng, cu, nh=2, dk=3, dv=4, gate_scale=1.0):
    T = int(cu[-1])
    q = rng.standard_normal((T, nh, dk)) / np.sqrt(dk)
    k = rng.standard_normal((T, nh, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, nh, dv))
    g = -gate_scale * np.log1p(np.exp(rng.standard_normal((T, nh))))  # -softplus: log of a decay in (0, 1)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, nh))))
    do = rng.standard_normal((T, nh, dv))
    return q, k, v, g, beta, do


CU = np.array([0, 4, 4, 11], dtype=np.int32)


def test_finite_differences_every_input():
    rng = np.random.default_rng(0)
    q, k, v, g, beta, do = _case(rng, CU)
    scale = 0.7
    grads = gdn.backward(q, k, v, g, beta, do, CU, scale)
    args = [q, k, v, g, beta]
    h = 1e-6
    for idx, (x, gx) in enumerate(zip(args, grads)):
        num = np.zeros_like(x)
        for pos in np.ndindex(x.shape):
            saved = x[pos]
            x[pos] = saved + h
            lp = np.sum(do * gdn.forward(*args, CU, scale))
            x[pos] = saved - h
            lm = np.sum(do * gdn.forward(*args, CU, scale))
            x[pos] = saved
            num[pos] = (lp - lm) / (2 * h)
        err = np.max(np.abs(num - gx)) / max(np.max(np.abs(num)), 1e-12)
        assert err < 1e-7, (idx, err)


def test_torch_autograd_through_the_recurrence():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    cu = np.array([0, 9, 9, 20], dtype=np.int32)
    q, k, v, g, beta, do = _case(rng, cu, nh=3, dk=5, dv=6)
    scale = 0.45
    ts = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v, g, beta)]
    tq, tk, tv, tg, tb = ts
    outs = []
    for a, b in zip(cu[:-1], cu[1:]):
        S = torch.zeros(3, 6, 5, dtype=torch.float64)  # the paper's S = H^T, [H, dv, dk]
        for t in range(int(a), int(b)):
            al = torch.exp(tg[t])
            eye = torch.eye(5, dtype=torch.float64)
            kk = tk[t][:, :, None] * tk[t][:, None, :]
            S = al[:, None, None] * S @ (eye - tb[t][:, None, None] * kk) + tb[t][:, None, None] * (
                tv[t][:, :, None] * tk[t][:, None, :])
            outs.append(scale * (S @ tq[t][:, :, None])[:, :, 0])
    o = torch.stack(outs)
    np.testing.assert_allclose(o.detach().numpy(), gdn.forward(q, k, v, g, beta, cu, scale), rtol=1e-12, atol=1e-12)
    (o * torch.tensor(do)).sum().backward()
    ours = gdn.backward(q, k, v, g, beta, do, cu, scale)
    for t, mine in zip(ts, ours):
        np.testing.assert_allclose(mine, t.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_zero_decay_keeps_only_the_current_token():
    # alpha = 0: H_t = beta_t k_t v_t^T, so o_t = scale beta_t <q_t, k_t> v_t.
    rng = np.random.default_rng(2)
    q, k, v, g, beta, _ = _case(rng, CU)
    g[:] = -np.inf
    o = gdn.forward(q, k, v, g, beta, CU, 0.9)
    want = 0.9 * beta[:, :, None] * np.sum(q * k, axis=-1)[:, :, None] * v
    np.testing.assert_allclose(o, want, rtol=1e-13, atol=1e-14)


def test_zero_beta_writes_nothing():
    rng = np.random.default_rng(3)
    q, k, v, g, beta, _ = _case(rng, CU)
    beta[:] = 0.0
    assert np.all(gdn.forward(q, k, v, g, beta, CU) == 0.0)


def test_orthogonal_keys_without_decay_is_causal_linear_attention():
    # With orthogonal keys the delta correction vanishes: e_t = beta_t v_t and
    # o_t = scale sum_{j <= t} beta_j <q_t, k_j> v_j within the segment.
    rng = np.random.default_rng(4)
    cu = np.array([0, 5, 8], dtype=np.int32)
    dk = 6
    q, k, v, g, beta, _ = _case(rng, cu, dk=dk)
    g[:] = 0.0
    basis = np.eye(dk)
    for a, b in zip(cu[:-1], cu[1:]):
        for t in range(a, b):
            k[t] = basis[(t - a) % dk] * 0.8
    o = gdn.forward(q, k, v, g, beta, cu, 1.3)
    for a, b in zip(cu[:-1], cu[1:]):
        for t in range(a, b):
            want = sum(beta[j][:, None] * np.sum(q[t] * k[j], -1)[:, None] * v[j] for j in range(a, t + 1))
            np.testing.assert_allclose(o[t], 1.3 * want, rtol=1e-12, atol=1e-13)


def test_one_repeated_unit_key_remembers_the_last_value():
    # alpha = beta = 1 and k_t = k (unit): the delta rule overwrites, H_t = k v_t^T.
    rng = np.random.default_rng(5)
    cu = np.array([0, 7], dtype=np.int32)
    q, k, v, g, beta, _ = _case(rng, cu)
    k[:] = k[0]
    g[:] = 0.0
    beta[:] = 1.0
    o = gdn.forward(q, k, v, g, beta, cu, 1.0)
    want = np.sum(q * k, axis=-1)[:, :, None] * v
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-13)


def test_decay_multiplies_from_the_token_after_the_write():
    # beta = 1 at the first token, 0 afterwards: H_t = (prod_{j=2..t} alpha_j) k_1 v_1^T.
    rng = np.random.default_rng(6)
    cu = np.array([0, 6], dtype=np.int32)
    q, k, v, g, beta, _ = _case(rng, cu)
    beta[:] = 0.0
    beta[0] = 1.0
    o = gdn.forward(q, k, v, g, beta, cu, 1.0)
    for t in range(6):
        decay = np.exp(np.sum(g[1:t + 1], axis=0))
        want = decay[:, None] * np.sum(q[t] * k[0], -1)[:, None] * v[0]
        np.testing.assert_allclose(o[t], want, rtol=1e-12, atol=1e-14)


def test_segments_are_isolated_and_empty_segments_change_nothing():
    rng = np.random.default_rng(7)
    cu = np.array([0, 5, 12, 20], dtype=np.int32)
    q, k, v, g, beta, do = _case(rng, cu)
    o = gdn.forward(q, k, v, g, beta, cu)
    grads = gdn.backward(q, k, v, g, beta, do, cu)
    # separate runs per segment give the same bits
    for a, b in zip(cu[:-1], cu[1:]):
        sub = [x[a:b] for x in (q, k, v, g, beta)]
        np.testing.assert_array_equal(gdn.forward(*sub, np.array([0, b - a], np.int32)), o[a:b])
    # perturbing the middle document leaves the others bit-identical
    q2, v2 = q.copy(), v.copy()
    q2[5:12] += 1.0
    v2[5:12] -= 2.0
    o2 = gdn.forward(q2, k, v2, g, beta, cu)
    np.testing.assert_array_equal(o2[:5], o[:5])
    np.testing.assert_array_equal(o2[12:], o[12:])
    # repeated boundaries (empty segments) anywhere change nothing
    cu_pad = np.array([0, 0, 5, 5, 5, 12, 20, 20], dtype=np.int32)
    np.testing.assert_array_equal(gdn.forward(q, k, v, g, beta, cu_pad), o)
    for x, y in zip(gdn.backward(q, k, v, g, beta, do, cu_pad), grads):
        np.testing.assert_array_equal(x, y)


def _chunked(q, k, v, g, beta, cu, scale, C):
    """The chunked (WY) form of the same recurrence, from the algebra: within
    a chunk, with gamma the running sum of g from the chunk start,
    (I + A) E = diag(beta) V - diag(beta e^gamma) K H0 with
    A_ij = beta_i e^(gamma_i - gamma_j) <k_i, k_j> (j < i), then
    O = diag(e^gamma) Q H0 scale + (tril(Q K^T) o Gamma) E scale and
    H1 = e^gamma_last H0 + (diag(e^(gamma_last - gamma)) K)^T E."""
    T, nh, dk = k.shape
    dv = v.shape[2]
    o = np.zeros((T, nh, dv))
    for a, b in zip(cu[:-1], cu[1:]):
        for h in range(nh):
            H0 = np.zeros((dk, dv))
            for c0 in range(int(a), int(b), C):
                c1 = min(int(b), c0 + C)
                K, V, Q = k[c0:c1, h], v[c0:c1, h], q[c0:c1, h]
                gam = np.cumsum(g[c0:c1, h])
                bt = beta[c0:c1, h]
                Gam = np.exp(gam[:, None] - gam[None, :])
                n = c1 - c0
                A = np.tril(bt[:, None] * Gam * (K @ K.T), -1)
                Tm = np.linalg.inv(np.eye(n) + A)
                W = Tm @ ((bt * np.exp(gam))[:, None] * K)
                U = Tm @ (bt[:, None] * V)
                E = U - W @ H0
                o[c0:c1, h] = scale * (np.exp(gam)[:, None] * (Q @ H0) + (np.tril(Q @ K.T) * np.tril(Gam)) @ E)
                H0 = np.exp(gam[-1]) * H0 + (np.exp(gam[-1] - gam)[:, None] * K).T @ E
    return o


@pytest.mark.parametrize("C", [1, 3, 4, 16])
def test_chunked_form_matches_the_recurrence(C):
    rng = np.random.default_rng(8)
    cu = np.array([0, 13, 13, 40, 47], dtype=np.int32)
    q, k, v, g, beta, _ = _case(rng, cu, nh=2, dk=8, dv=5, gate_scale=0.3)
    want = gdn.forward(q, k, v, g, beta, cu, 0.35)
    np.testing.assert_allclose(_chunked(q, k, v, g, beta, cu, 0.35, C), want, rtol=1e-9, atol=1e-11)


def test_checkpointed_backward_matches_across_checkpoint_sizes(monkeypatch):
    # The backward recomputes states between checkpoints; its result must not
    # depend on where the checkpoints fall.
    rng = np.random.default_rng(9)
    cu = np.array([0, 23, 30], dtype=np.int32)
    q, k, v, g, beta, do = _case(rng, cu)
    ref = gdn.backward(q, k, v, g, beta, do, cu)
    monkeypatch.setattr(gdn, "CHECKPOINT", 5)
    for x, y in zip(gdn.backward(q, k, v, g, beta, do, cu), ref):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-14)
