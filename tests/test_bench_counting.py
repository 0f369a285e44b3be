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
