"""The benchmark's counting rules, checked on the CPU against the oracle and
the definitions they restate: unmasked pairs (the FLOP count's base), the
algorithmic HBM bytes of a step, and the pair counts the input generator
gives for the named 16K workloads."""
import numpy as np
import pytest

import bench
import oracle
from varlen_sliding_window_gb300 import synth


@pytest.mark.parametrize("name", ["tiny_global", "tiny_w64", "ctx512_global", "ctx4096_w512", "ctx4096_global"])
def test_closed_form_pairs_equal_oracle_masks(name):
    wl = synth.workloads()[name]
    cu = wl.cu_seqlens()
    assert bench.unmasked_pairs(cu, wl.window_left) == oracle.unmasked_pairs(cu, wl.window_left)


def test_pair_counts_of_the_named_workloads():
    # Values the generator reproduces for doc seed 0 (scratch simulation of the recipe).
    wls = synth.workloads()
    assert bench.unmasked_pairs(wls["tiny_global"].cu_seqlens(), -1) == 11501
    assert bench.unmasked_pairs(wls["tiny_w64"].cu_seqlens(), 64) == 10406
    assert abs(bench.unmasked_pairs(wls["ctx512_global"].cu_seqlens(), -1) - 3.55e6) < 0.01e6
    assert abs(bench.unmasked_pairs(wls["ctx4096_w512"].cu_seqlens(), 512) - 5.87e6) < 0.01e6
    assert abs(bench.unmasked_pairs(wls["ctx4096_global"].cu_seqlens(), -1) - 11.82e6) < 0.01e6


def test_algorithmic_bytes_of_a_16k_step():
    wl = synth.workloads()["ctx512_global"]
    mib = 1024 * 1024
    # forward 80.5 MiB (q, k, v, out, lse) + backward 161.5 MiB (q, k, v, out,
    # dout, lse read; dq, dk, dv written; D written and read).
    assert bench.algorithmic_bytes(wl) == int((80.5 + 161.5) * mib)


def test_flop_rule():
    wl = synth.workloads()["ctx4096_global"]
    pairs = bench.unmasked_pairs(wl.cu_seqlens(), -1)
    # 4 d Hq pairs (forward) x 3.5 (forward + 2.5 x forward for the backward)
    flops = 4 * 128 * 8 * pairs * 3.5
    r = bench.roofs(wl, pairs, 1.0, 1900.0, 6800.0, 2070.0)
    assert np.isclose(r["tensor"]["achieved_tflops"], flops / 1e-3 / 1e12)
    assert r["exp"]["count"] == 3 * pairs * 8


def test_gdn_flop_count_lists_every_product():
    # One segment of 64 + 1 tokens, one head of width 128: the forward's
    # products written out shape by shape (M x K x N, 2 MKN flops each).
    d = 128

    def prods(n):
        fwd = [(n, d, n), (n, d, n), (n, n, d), (n, n, d),       # K K^T, Q K^T, W, U
               (n, d, d), (n, d, d), (n, n, d), (d, n, d)]       # W H, Q H, Aq E, K^T E
        rec = [(n, d, n), (n, d, n), (n, n, d), (n, n, d), (n, d, d), (d, n, d)]
        state = [(n, n, d), (n, d, d), (d, n, d), (d, n, d)]     # Aq^T dO, K dH, Q^T G, W^T dE
        loc_h = [(n, d, n), (n, d, n), (n, d, d), (n, n, d), (n, d, d), (n, d, d), (n, n, d), (n, d, d),
                 (n, d, d)]
        loc_wy = [(n, d, n)] * 3 + [(n, n, d)] * 4 + [(n, n, n)] * 2
        f = sum(2 * a * b * c for a, b, c in fwd)
        b = sum(2 * a * b * c for a, b, c in rec + state + loc_h + loc_wy)
        return f, b

    f64, b64 = prods(64)
    f1, b1 = prods(1)
    ff, fb = bench.gdn_flops(np.array([0, 65], dtype=np.int32), 1, d)
    assert ff == f64 + f1 and fb == b64 + b1
    ff2, fb2 = bench.gdn_flops(np.array([0, 65, 65], dtype=np.int32), 3, d)
    assert ff2 == 3 * ff and fb2 == 3 * fb


def test_kda_flop_count_lists_every_product():
    d = 128

    def prods(n):
        qk = [(n, d, n)] * 2                                                   # K K^T, Q K^T (10 of 16 blocks)
        fwd_rest = [(n, n, d), (n, n, d), (n, d, d), (n, d, d), (n, n, d), (d, n, d)]  # W, U, W H, QB H, Aq E, KC^T E
        rec_rest = [(n, n, d), (n, n, d), (n, d, d), (d, n, d)]               # W, U, W H, KC^T E
        state = [(n, n, d), (n, d, d), (d, n, d), (d, n, d)]
        loc_h = [(n, d, n), (n, d, d), (n, d, d), (n, d, d)]                   # dO E^T, dO H0^T, dE H0^T, E dH1^T
        loc_wy = [(n, d, n)] * 2 + [(n, n, n)] * 2 + [(n, n, d)] * 2
        f = sum(2 * a * b * c for a, b, c in fwd_rest) + sum(2 * a * b * c for a, b, c in qk) * 10 / 16
        b = (sum(2 * a * b * c for a, b, c in rec_rest + state + loc_h + loc_wy)
             + sum(2 * a * b * c for a, b, c in qk) * 10 / 16 + 4 * d * n * n)
        return f, b

    f64, b64 = prods(64)
    ff, fb = bench.gdn_flops(np.array([0, 64], dtype=np.int32), 1, d, per_channel=True)
    assert ff == f64 and fb == b64
