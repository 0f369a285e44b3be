"""The per-segment parity check itself, on the CPU: it accepts results within
the tolerance and flags a single wrong segment that the whole-tensor norm
would let through."""
import numpy as np
import pytest

import oracle

from helpers import TOL_GRAD, assert_per_segment, rel_l2


def test_per_segment_check_flags_one_wrong_segment():
    rng = np.random.default_rng(0)
    cu = np.array([0, 3, 40, 1000, 3000], dtype=np.int32)
    T = int(cu[-1])
    q, k, v, do = (rng.standard_normal((T, h, 16)) for h in (4, 2, 2, 4))
    dq, _, _ = oracle.backward(do, q, k, v, cu, -1, 0.25)
    noisy = dq * (1 + 1e-3 * rng.standard_normal(dq.shape))
    assert_per_segment(noisy, dq, cu, TOL_GRAD, "dq")
    bad = noisy.copy()
    bad[3:40] *= 1.025  # one 37-token segment off by 2.5 %
    assert rel_l2(bad, dq) < TOL_GRAD  # invisible in the norm of the whole tensor
    with pytest.raises(AssertionError):
        assert_per_segment(bad, dq, cu, TOL_GRAD, "dq")
    short = noisy.copy()
    short[0:3] = 0.0  # a wrong 3-token segment
    with pytest.raises(AssertionError):
        assert_per_segment(short, dq, cu, TOL_GRAD, "dq")
