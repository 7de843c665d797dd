"""Backward parity: dQ/dK/dV from the CUDA path (B1 preprocess, B2 main
kernel, B3 finalise, through fa_backward) against the oracle's gradients
computed with P materialised, on the same seeded bf16 inputs."""

import math

import numpy as np
import pytest
import torch

import oracle
from parity import GRAD_REL, check_forward, check_grads, nan_backward, nan_forward
from workloads import WORKLOADS, as_f64, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_27_gb300 import _build
    _build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_fwd_bwd(inp, causal, scale):
    import exact_attention_27_gb300 as fa
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = nan_forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = nan_backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    return o, lse, (dq, dk, dv)


def bwd_vs_oracle(inp, causal, scale, check_fwd=True):
    o, lse, grads = run_fwd_bwd(inp, causal, scale)
    f = {n: as_f64(inp[n]) for n in ("q", "k", "v", "do")}
    if check_fwd:
        o_ref, l_ref = oracle.attention_forward(f["q"], f["k"], f["v"], scale, causal)
        check_forward(o, lse, o_ref, l_ref, "forward")
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], scale, causal)
    check_grads(grads, ref, "backward")
    return grads


def test_causal_train_n4096_d64():
    w = WORKLOADS["causal_train_n4096_d64"]
    bwd_vs_oracle(workload_inputs(w), w.causal, w.scale)


@pytest.mark.parametrize("N", [1, 5, 70, 128, 129, 257, 600])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(N, d, causal):
    inp = make_inputs(1, 2, 2, N, d, seed=N * 3 + d, with_grad=True)
    bwd_vs_oracle(inp, causal, 1.0 / math.sqrt(d))


@pytest.mark.parametrize("G", [2, 4])
@pytest.mark.parametrize("d", [64, 128])
def test_grouped_query_heads(G, d):
    """dK and dV of a shared head sum over the G query heads that read it."""
    inp = make_inputs(2, 8, 8 // G, 300, d, seed=70 + G + d, with_grad=True)
    bwd_vs_oracle(inp, True, 1.0 / math.sqrt(d))


@pytest.mark.parametrize("d", [64, 96, 128])
@pytest.mark.parametrize("N", [200, 513])
def test_grouped_query_heads_non_causal(d, N):
    """Non-causal: every key tile sees every query tile of all G heads of its
    group, so dK and dV sum over the whole group at every key."""
    inp = make_inputs(2, 8, 2, N, d, seed=700 + N + d, with_grad=True)
    bwd_vs_oracle(inp, False, 1.0 / math.sqrt(d))


@pytest.mark.parametrize("N", [1, 70, 129, 600])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_96(N, causal):
    """d = 96 through the padded 128-column kernels: gradients of the 96 real
    columns against the oracle; GQA so that dK/dV sum over two heads."""
    inp = make_inputs(1, 4, 2, N, 96, seed=N + 960, with_grad=True)
    bwd_vs_oracle(inp, causal, 1.0 / math.sqrt(96))


@pytest.mark.parametrize("N", [1, 5, 63, 64, 65, 129, 200, 600])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_256(N, causal):
    """d = 256: dK and dV from 64-key tiles with the accumulators held
    transposed, then dQ from the query-tile kernel; GQA so that dK/dV sum over
    two heads.  Ragged lengths around the 64-key and 128-query tiles."""
    inp = make_inputs(1, 4, 2, N, 256, seed=N + 2560, with_grad=True)
    bwd_vs_oracle(inp, causal, 1.0 / math.sqrt(256))


@pytest.mark.parametrize("G", [1, 4])
def test_head_dim_256_grouped_query_heads(G):
    inp = make_inputs(2, 8, 8 // G, 300, 256, seed=2570 + G, with_grad=True)
    bwd_vs_oracle(inp, True, 1.0 / math.sqrt(256))


def test_head_dim_256_large_scores():
    """Scores spanning many log2 units (Q scaled by 3): P rebuilt from L must
    stay exact.  Gradients only: with the softmax this sharp the forward's
    absolute O error sits at the edge of the N(0,1)-input bound (bf16 P and O
    times |v| up to ~5), which the forward tests cover on their own inputs."""
    inp = make_inputs(1, 2, 1, 700, 256, seed=2580, with_grad=True)
    inp["q"] = (inp["q"].float() * 3.0).to(torch.bfloat16)
    bwd_vs_oracle(inp, True, 0.25, check_fwd=False)


def test_head_dim_256_both_entry_points_agree_bit_for_bit():
    """At d = 256 fa_backward runs the same two atomic-free kernels as
    fa_backward_deterministic: identical bits, and run to run."""
    import exact_attention_27_gb300 as fa
    inp = make_inputs(1, 8, 2, 777, 256, seed=2590, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = nan_forward(q, k, v, causal=True)
    g1 = nan_backward(q, k, v, o, lse, do, causal=True)
    g2 = nan_backward(q, k, v, o, lse, do, causal=True, deterministic=True)
    g3 = nan_backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    for a, b, c in zip(g1, g2, g3):
        assert torch.equal(a, b) and torch.equal(a, c)


def test_d128_causal_mid_size():
    inp = make_inputs(1, 4, 4, 1024, 128, seed=123, with_grad=True)
    bwd_vs_oracle(inp, True, 1.0 / math.sqrt(128))


@pytest.mark.parametrize("d", [64, 96, 128, 256])
def test_preprocess_row_dot(d):
    """B1 alone: D = rowsum(dO o O) against the oracle's row_dot."""
    import exact_attention_27_gb300 as fa
    inp = make_inputs(3, 5, 5, 333, d, seed=d, with_grad=True)
    o, do = inp["q"].cuda(), inp["do"].cuda()
    D = torch.full(o.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_backward_preprocess(o, do, D)
    torch.cuda.synchronize()
    ref = oracle.row_dot(as_f64(inp["do"]), as_f64(inp["q"]))
    mag = oracle.row_dot(np.abs(as_f64(inp["do"])), np.abs(as_f64(inp["q"])))
    # products of bf16 values are exact in fp32; d additions in fp32
    assert np.all(np.abs(D.cpu().numpy() - ref) <= d * 2.0 ** -24 * mag + 1e-6)


def test_gradients_do_not_depend_on_output_buffers_contents():
    """Outputs are fully written: garbage in dq/dk/dv beforehand changes nothing."""
    import exact_attention_27_gb300 as fa
    inp = make_inputs(1, 2, 1, 333, 64, seed=8, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = nan_forward(q, k, v, causal=True)
    outs = []
    for fill in (0.0, float("nan")):
        dq = torch.full_like(q, fill)
        dk = torch.full_like(k, fill)
        dv = torch.full_like(v, fill)
        fa.fa_backward(q, k, v, o, lse, do, dq, dk, dv, 0.125, True)
        torch.cuda.synchronize()
        outs.append((dq.float(), dk.float(), dv.float()))
    for a, b in zip(*outs):
        assert torch.isfinite(b).all()
        assert torch.allclose(a, b, atol=1e-2, rtol=0)


def run_deterministic(inp, causal, scale):
    import exact_attention_27_gb300 as fa
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = nan_forward(q, k, v, causal=causal, scale=scale)
    grads = nan_backward(q, k, v, o, lse, do, causal=causal, scale=scale,
                                  deterministic=True)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    return (q, k, v, do, o, lse), grads


@pytest.mark.parametrize("shape", [
    (2, 8, 8, 4096, 64, True),      # the training workload
    (1, 2, 2, 70, 64, False),
    (1, 2, 2, 257, 128, True),
    (2, 8, 2, 300, 64, True),       # grouped-query heads
    (1, 4, 1, 513, 128, False),
    (1, 2, 2, 1, 64, True),
    (1, 4, 2, 333, 96, True),
    (1, 2, 1, 200, 96, False),
    (1, 4, 2, 333, 256, True),
    (1, 2, 1, 200, 256, False),
])
def test_deterministic_backward_against_the_oracle(shape):
    B, Hq, Hkv, N, d, causal = shape
    inp = make_inputs(B, Hq, Hkv, N, d, seed=90 + N, with_grad=True)
    scale = 1.0 / math.sqrt(d)
    _, grads = run_deterministic(inp, causal, scale)
    f = {n: as_f64(inp[n]) for n in ("q", "k", "v", "do")}
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], scale, causal)
    check_grads(grads, ref, "deterministic backward")


@pytest.mark.parametrize("d,G", [(64, 1), (128, 4)])
def test_deterministic_backward_is_bitwise_reproducible(d, G):
    """Two runs give identical bits; dK and dV also equal the single-kernel
    path's bit for bit (same products in the same order)."""
    import exact_attention_27_gb300 as fa
    inp = make_inputs(2, 8, 8 // G, 1000, d, seed=5, with_grad=True)
    scale = 1.0 / math.sqrt(d)
    (q, k, v, do, o, lse), g1 = run_deterministic(inp, True, scale)
    g2 = nan_backward(q, k, v, o, lse, do, causal=True, scale=scale, deterministic=True)
    g3 = nan_backward(q, k, v, o, lse, do, causal=True, scale=scale)
    torch.cuda.synchronize()
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
    assert torch.equal(g1[1], g3[1]) and torch.equal(g1[2], g3[2])


@pytest.mark.parametrize("B,Hq,Hkv,N,d,det", [
    (2, 16, 16, 4096, 128, False),   # the d = 128 backward timed beside the step
    (2, 16, 16, 4096, 96, False),    # the d = 96 one
    (1, 8, 2, 4096, 128, False),     # grouped-query heads at full length
    (2, 16, 16, 4096, 128, True),    # the deterministic path at the same size
    (1, 2, 2, 32768, 64, False),     # long sequence: 256 query tiles for the first key tile
    (1, 2, 2, 32768, 64, True),      # and the deterministic path there
    (2, 16, 16, 4096, 256, False),   # the d = 256 backward timed beside the step
    (1, 8, 2, 8192, 256, True),      # d = 256, grouped-query heads, longer sequence
])
def test_full_size_backward_sampled(B, Hq, Hkv, N, d, det):
    """Full-size causal backward against the oracle on two 256-row query
    blocks (the first and the last).  Under the causal mask the last 256 keys
    are seen only by the last 256 queries, so the oracle's backward of that
    block gives their dK and dV completely; dQ of both blocks is complete
    too.  Bounds: the forward's, and 5e-2 x max |reference| over each sampled
    gradient block."""
    import exact_attention_27_gb300 as fa
    inp = make_inputs(B, Hq, Hkv, N, d, seed=11, with_grad=True)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = nan_forward(q, k, v, causal=True, scale=scale)
    dq, dk, dv = nan_backward(q, k, v, o, lse, do, causal=True, scale=scale,
                              deterministic=det)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    f = {n: as_f64(inp[n]) for n in ("q", "k", "v", "do")}
    blk = 256
    for r0 in (0, N - blk):
        rows = slice(r0, r0 + blk)
        o_ref, l_ref = oracle.attention_forward(f["q"][:, :, rows], f["k"], f["v"], scale, True,
                                                q_offset=r0)
        check_forward(o[:, :, rows], lse[:, :, rows], o_ref, l_ref, f"forward rows {r0}..")
        dq_ref, dk_ref, dv_ref = oracle.attention_backward(f["q"][:, :, rows], f["k"], f["v"],
                                                           f["do"][:, :, rows], scale, True,
                                                           q_offset=r0)
        got, ref = [dq[:, :, rows]], [dq_ref]
        if r0 == N - blk:
            got += [dk[:, :, rows], dv[:, :, rows]]
            ref += [dk_ref[:, :, rows], dv_ref[:, :, rows]]
        for g, r in zip(got, ref):
            g = g.float().cpu().numpy().astype(np.float64)
            assert np.isfinite(g).all()
            err = np.abs(g - r).max()
            assert err <= GRAD_REL * np.abs(r).max(), f"rows {r0}..: err {err:.3e}"


@pytest.mark.parametrize("d", [64, 96, 128, 256])
@pytest.mark.parametrize("det", [False, True])
def test_many_heads_tiny_sequence(d, det):
    """B x H_q = 4096 heads of 17 positions, GQA 2: every CTA holds one
    partial tile (and the forward's second tile of a pair lies wholly past
    N).  Forward and gradients, every row, against the oracle."""
    import exact_attention_27_gb300 as fa
    B, Hq, Hkv, N = 64, 64, 32, 17
    inp = make_inputs(B, Hq, Hkv, N, d, seed=d + det, with_grad=True)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = nan_forward(q, k, v, causal=True, scale=scale)
    grads = nan_backward(q, k, v, o, lse, do, causal=True, scale=scale,
                         deterministic=det)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    f = {n: as_f64(inp[n]) for n in ("q", "k", "v", "do")}
    o_ref, l_ref = oracle.attention_forward(f["q"], f["k"], f["v"], scale, True)
    check_forward(o, lse, o_ref, l_ref, "many heads")
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], scale, True)
    check_grads(grads, ref, "many heads")
