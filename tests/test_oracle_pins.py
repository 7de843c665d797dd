"""The CPU oracle against the pages' worked examples, closed forms, invariants,
an exact-summation evaluation, finite differences and a library routine."""

import math

import pytest

import oracle
from oracle.online_softmax import naive_block_average, online_softmax_row
from oracle_pins import ALL_PINS, golden


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle.load())


def test_two_block_note_blockwise():
    """paweldubiel.com note: block results 0 and 1, exact 0.75, naive mean 0.5."""
    g = golden()["two_block_note"]
    s = [0.0, 0.0, math.log(3.0), math.log(3.0)]
    out, lse, trace = online_softmax_row(s, g["values"], g["block"])
    assert abs(out - g["exact_result"]) < 1e-15
    assert abs(lse - math.log(8.0)) < 1e-15
    # the per-block normalised results the note quotes
    assert [t["o"] / t["l"] for t in trace][0] == g["block_results"][0]
    blk2 = online_softmax_row(s[2:], g["values"][2:], 2)[0]
    assert abs(blk2 - g["block_results"][1]) < 1e-15
    naive = naive_block_average(s, g["values"], g["block"])
    assert naive == g["naive_block_mean"]
    assert naive != g["exact_result"]


def test_four_scores_trace():
    """Page 1: blocks [1,3], [2,4]: m1=3, l1~1.135, alpha~0.368, m2=4, l2~1.553."""
    g = golden()["four_scores"]
    _, _, trace = online_softmax_row(g["scores"], [0.0] * 4, g["block"])
    tol = 0.5e-3 + 1e-12
    assert trace[0]["m"] == g["block1"]["m"] and trace[0]["alpha"] is None
    assert abs(trace[0]["l"] - g["block1"]["l"]) <= tol
    assert trace[1]["m"] == g["block2"]["m"]
    assert abs(trace[1]["alpha"] - g["block2"]["alpha"]) <= tol
    assert abs(trace[1]["l"] - g["block2"]["l"]) <= tol


def test_figure_7_9_trace():
    """Fig. 7.9: alpha 0.368 where the record rises (blocks 2 and 4), o/l = 5.257."""
    g = golden()["figure_7_9"]
    out, _, trace = online_softmax_row(g["scores"], g["values"], g["block"])
    assert abs(out - g["result"]) <= 0.5e-3
    for n, t in enumerate(trace, start=1):
        if n in g["record_rises_at_blocks"]:
            assert abs(t["alpha"] - g["alpha_when_record_rises"]) <= 0.5e-3
        elif n > 1:
            assert t["alpha"] == 1.0


def test_flop_and_byte_convention():
    """Page 1's unfused balance at N=8192, d=64 and its FLOP counts, recomputed.

    These fix the FLOP convention the benchmark uses (4 N^2 d forward,
    10 N^2 d backward with the recompute)."""
    g = golden()["cost_unfused_n8192_d64"]
    N, d = g["N"], g["d"]
    assert round(N * N / 1e6) == g["score_elements_million"]
    assert round(N * N * 2 / 1e6) == g["score_matrix_MB_fp16"]
    matmul_flop = 2 * (2 * N * N * d)
    assert abs(matmul_flop / 1e9 - g["gflop_approx"]) < 0.5   # plus a few softmax ops / element
    bytes_ = 4 * N * N * 2 + 4 * N * d * 2                     # S, P written + re-read; Q, K, V, O
    assert abs(bytes_ / 1e6 - g["MB_approx"]) < 1.0
    assert round(matmul_flop / bytes_) == g["flop_per_byte"]
    for dd, want in ((64, g["matmul_intensity_d64"]), (128, g["matmul_intensity_d128"])):
        intensity = 2 * N * N * dd / (2 * N * N + 2 * N * dd * 2)
        assert round(intensity) == want
    fc = golden()["flop_counts"]
    from workloads import Workload
    w = Workload("x", 1, 1, 1, N, d, False, True)
    assert w.fwd_flops() == fc["forward_coeff"] * N * N * d
    assert w.bwd_flops() == fc["backward_recompute_coeff"] * N * N * d
    # a quarter more on the backward, a sixth more on the total
    assert fc["backward_recompute_coeff"] / fc["backward_standard_coeff"] == 1.25
    tot_std = fc["forward_coeff"] + fc["backward_standard_coeff"]
    tot_fa = fc["forward_coeff"] + fc["backward_recompute_coeff"]
    assert abs(tot_fa / tot_std - 7 / 6) < 1e-12
    wc = Workload("x", 1, 1, 1, N, d, True, True)
    assert wc.fwd_flops() == w.fwd_flops() / 2


def test_oracle_rejects_bad_shapes():
    import numpy as np
    orc = oracle.load()
    q = np.zeros((1, 3, 4, 2))
    k = np.zeros((1, 2, 4, 2))
    with pytest.raises(RuntimeError):
        orc.forward(q, k, k, 1.0, False)  # 3 query heads over 2 K/V heads
