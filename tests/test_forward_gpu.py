"""Forward parity: the CUDA path through the C ABI against the CPU oracle on
the same seeded bf16 inputs."""

import math

import numpy as np
import pytest
import torch

import oracle
from parity import check_forward, forward_vs_oracle, gpu_forward
from workloads import WORKLOADS, as_f64, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_27_gb300 import _build
    _build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_single_head_n256():
    w = WORKLOADS["single_head_n256"]
    forward_vs_oracle(workload_inputs(w), w.causal, w.scale)


def test_worked_example_through_the_boundary():
    """Scores [0, 0, ln3, ln3] and values [0, 0, 1, 1] give 0.75 in every row
    (paweldubiel.com note); q_i = e_0, k_j = (0,0,1,1)_j e_0, scale = ln 3."""
    d = 64
    q = torch.zeros(1, 1, 4, d, dtype=torch.bfloat16)
    q[..., 0] = 1.0
    k = torch.zeros(1, 1, 4, d, dtype=torch.bfloat16)
    k[0, 0, 2:, 0] = 1.0
    v = k.clone()
    scale = float(np.float32(math.log(3.0)))
    inp = {"q": q, "k": k, "v": v}
    o, lse = gpu_forward(inp, False, scale)
    o = o.float().cpu()
    assert torch.all(o[0, 0, :, 0] == 0.75)
    assert torch.all(o[0, 0, :, 1:] == 0.0)
    assert torch.allclose(lse.cpu(), torch.full((1, 1, 4), math.log(8.0)), atol=1e-3)
    forward_vs_oracle(inp, False, scale)


def test_causal_first_row_returns_v0_exactly():
    inp = make_inputs(2, 4, 2, 300, 64, seed=11)
    o, lse = gpu_forward(inp, True, 0.125)
    G = 2
    for h in range(4):
        assert torch.equal(o[:, h, 0].cpu(), inp["v"][:, h // G, 0])
    ref = 0.125 * (inp["q"][:, :, 0].double() *
                   inp["k"].repeat_interleave(G, 1)[:, :, 0].double()).sum(-1)
    assert torch.allclose(lse[:, :, 0].cpu().double(), ref, atol=1e-4)


@pytest.mark.parametrize("N", [1, 4, 70, 128, 129, 257, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(N, d, causal):
    inp = make_inputs(1, 2, 1, N, d, seed=N + d)
    forward_vs_oracle(inp, causal, 1.0 / math.sqrt(d))


@pytest.mark.parametrize("G", [1, 2, 4])
def test_grouped_query_heads(G):
    inp = make_inputs(2, 8, 8 // G, 384, 128, seed=40 + G)
    forward_vs_oracle(inp, True, 1.0 / math.sqrt(128))


def test_large_scores_and_rescaling():
    """Scores spanning hundreds of log2 units exercise the lazy rescale path."""
    inp = make_inputs(1, 2, 2, 640, 64, seed=5)
    inp["q"] = (inp["q"].float() * 6.0).to(torch.bfloat16)
    forward_vs_oracle(inp, True, 1.0)
    forward_vs_oracle(inp, False, 1.0)


def test_causal_n4096_d64_full():
    w = WORKLOADS["causal_n4096_d64"]
    forward_vs_oracle(workload_inputs(w), w.causal, w.scale)


def _sampled(w, n_rows, seed):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, w.N - 1],
                                     rng.integers(0, w.N, n_rows)]))
    return rows


@pytest.mark.parametrize("name", ["causal_n8192_d128", "causal_gqa_n16384_d128"])
def test_full_size_sampled_rows(name):
    """Full-size workloads in the benchmark's launch configuration: every head,
    a seeded sample of query rows plus the tile edges, against the oracle."""
    w = WORKLOADS[name]
    inp = workload_inputs(w)
    rows = _sampled(w, 24, seed=3)
    (_, _, _), (o, lse) = forward_vs_oracle(inp, w.causal, w.scale, rows=rows)


def test_deterministic():
    inp = make_inputs(1, 4, 2, 777, 128, seed=9)
    o1, l1 = gpu_forward(inp, True, 0.1)
    o2, l2 = gpu_forward(inp, True, 0.1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_selftest_timeout_is_reported_and_device_stays_usable():
    import exact_attention_27_gb300 as fa
    assert fa.fa_last_device_error() == 0
    fa.fa_selftest_wait_timeout(20)
    assert fa.fa_last_device_error() == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.fa_last_device_error() == 0  # cleared
    w = WORKLOADS["single_head_n256"]
    forward_vs_oracle(workload_inputs(w), w.causal, w.scale)
