"""Forward parity: the CUDA path through the C ABI against the CPU oracle on
the same seeded bf16 inputs."""

import math

import numpy as np
import pytest
import torch

import oracle
from parity import (check_forward, forward_every_element, forward_vs_oracle, gpu_forward,
                    nan_forward, nan_outputs)
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


@pytest.mark.parametrize("N", [1, 70, 128, 257, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_96(N, causal):
    """d = 96: tiles padded to 128 columns (zero-filled), 96 stored."""
    inp = make_inputs(1, 4, 2, N, 96, seed=N + 96)
    forward_vs_oracle(inp, causal, 1.0 / math.sqrt(96))


def test_head_dim_96_query_offset():
    import exact_attention_27_gb300 as fa
    inp = make_inputs(2, 4, 1, 200, 96, seed=960, Nk=713)
    scale = 1.0 / math.sqrt(96)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = nan_forward(q, k, v, causal=True, scale=scale, q_offset=513)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    o_ref, l_ref = oracle.attention_forward(as_f64(inp["q"]), as_f64(inp["k"]), as_f64(inp["v"]),
                                            scale, True, q_offset=513)
    check_forward(o, lse, o_ref, l_ref, "d96 offset")


@pytest.mark.parametrize("N", [1, 63, 64, 65, 200, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_256(N, causal):
    """d = 256: one 128-row query tile per CTA, 64-key tiles, S double-buffered."""
    inp = make_inputs(1, 4, 2, N, 256, seed=N + 256)
    forward_vs_oracle(inp, causal, 1.0 / math.sqrt(256))


def test_head_dim_256_rescaling_and_many_tiles():
    """Large scores over 48 key tiles exercise the lazy rescale of the 256-column O."""
    inp = make_inputs(2, 2, 1, 3000, 256, seed=2560)
    inp["q"] = (inp["q"].float() * 4.0).to(torch.bfloat16)
    forward_vs_oracle(inp, True, 0.25)


@pytest.mark.parametrize("Nq,Nk,off,causal", [(1, 70, 69, True), (100, 513, 413, True),
                                              (128, 1000, 0, False), (300, 377, 77, True)])
def test_head_dim_256_query_offset(Nq, Nk, off, causal):
    import exact_attention_27_gb300 as fa
    inp = make_inputs(1, 4, 2, Nq, 256, seed=Nq + Nk + 256, Nk=Nk)
    scale = 1.0 / math.sqrt(256)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = nan_forward(q, k, v, causal=causal, scale=scale, q_offset=off)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    o_ref, l_ref = oracle.attention_forward(as_f64(inp["q"]), as_f64(inp["k"]), as_f64(inp["v"]),
                                            scale, causal, q_offset=off)
    check_forward(o, lse, o_ref, l_ref, f"d256 offset {off}")


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


@pytest.mark.parametrize("name", ["causal_n8192_d128", "causal_gqa_n16384_d128"])
def test_full_size_every_element(name):
    """The two d = 128 forward targets (B4 H16 N8192 and GQA B1 Hq32 Hkv8
    N16384) at full size, in the launch configuration the benchmark times
    (per-shape tile size, launch order and head grouping), into NaN-filled
    outputs: every element of O and L against the oracle, which is evaluated
    in blocks of query rows."""
    import exact_attention_27_gb300 as fa
    w = WORKLOADS[name]
    inp = workload_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = nan_outputs(q)
    fa.fa_forward(q, k, v, o, lse, w.scale, w.causal)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    del q, k, v
    forward_every_element(inp, w.causal, w.scale, o, lse, what=name)


def _tile_rows(N, seed):
    """The first and last row of every 128-row query tile, plus one row at a
    seeded offset inside each tile."""
    rng = np.random.default_rng(seed)
    starts = np.arange(0, N, 128)
    ends = np.minimum(starts + 127, N - 1)
    inner = np.minimum(starts + rng.integers(1, 127, starts.size), N - 1)
    return np.unique(np.concatenate([starts, ends, inner]))


@pytest.mark.parametrize("name", ["causal_n8192_d96", "causal_n8192_d256",
                                  "causal_gqa_n16384_d256"])
def test_full_size_every_tile_and_two_whole_heads(name):
    """Full-size d = 96 and d = 256 workloads in the benchmark's launch
    configuration, into NaN-filled outputs: every element finite (so written),
    three rows of every 128-row query tile of every head against the oracle,
    and every row of two whole heads (the first head of the first batch and
    the last head of the last batch)."""
    import exact_attention_27_gb300 as fa
    w = WORKLOADS[name]
    inp = workload_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = nan_outputs(q)
    fa.fa_forward(q, k, v, o, lse, w.scale, w.causal)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    del q, k, v
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    rows = _tile_rows(w.N, seed=w.d)
    o_ref, l_ref = oracle.attention_forward(as_f64(inp["q"]), as_f64(inp["k"]),
                                            as_f64(inp["v"]), w.scale, w.causal, rows=rows)
    check_forward(o[:, :, rows], lse[:, :, rows], o_ref, l_ref, f"{name} tile rows")
    G = w.Hq // w.Hkv
    for b, h in ((0, 0), (w.B - 1, w.Hq - 1)):
        head = {"q": inp["q"][b:b + 1, h:h + 1], "k": inp["k"][b:b + 1, h // G:h // G + 1],
                "v": inp["v"][b:b + 1, h // G:h // G + 1]}
        forward_every_element(head, w.causal, w.scale, o[b:b + 1, h:h + 1],
                              lse[b:b + 1, h:h + 1], block_rows=512, what=f"{name} head {b},{h}")


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


@pytest.mark.parametrize("Nq,Nk,off,causal,d,Hq,Hkv", [
    (1, 70, 69, True, 64, 2, 2),        # one query against 70 positions (the decode case)
    (1, 70, 0, True, 64, 2, 2),         # ... that sees only key 0
    (1, 70, 69, False, 64, 2, 1),
    (128, 1000, 872, True, 64, 4, 2),   # prefill continuing a cache
    (300, 377, 77, True, 128, 2, 2),    # offset not a multiple of the tile
    (257, 300, 0, True, 64, 2, 2),      # top-left alignment, N_q < N_kv
    (100, 513, 413, False, 128, 4, 1),
    (64, 4096, 4032, True, 128, 8, 2),
])
def test_query_offset_against_the_oracle(Nq, Nk, off, causal, d, Hq, Hkv):
    import exact_attention_27_gb300 as fa
    inp = make_inputs(1, Hq, Hkv, Nq, d, seed=Nq + Nk, Nk=Nk)
    scale = 1.0 / math.sqrt(d)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = nan_forward(q, k, v, causal=causal, scale=scale, q_offset=off)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    o_ref, l_ref = oracle.attention_forward(as_f64(inp["q"]), as_f64(inp["k"]), as_f64(inp["v"]),
                                            scale, causal, q_offset=off)
    check_forward(o, lse, o_ref, l_ref, f"offset {off}")


def test_offset_rows_equal_rows_of_the_full_forward():
    """Rows o..o+n-1 computed as queries with offset o match those rows of the
    same-sequence causal forward bit for bit (each row's arithmetic is the same)."""
    import exact_attention_27_gb300 as fa
    inp = make_inputs(2, 4, 2, 700, 64, seed=77)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o_full, l_full = nan_forward(q, k, v, causal=True, scale=0.125)
    for off, n in ((0, 128), (100, 300), (699, 1), (513, 187)):
        qs = q[:, :, off:off + n].contiguous()
        o, lse = nan_forward(qs, k, v, causal=True, scale=0.125, q_offset=off)
        torch.cuda.synchronize()
        assert torch.equal(o, o_full[:, :, off:off + n]), off
        assert torch.equal(lse, l_full[:, :, off:off + n]), off


def test_forward_ex_with_equal_lengths_is_forward():
    import exact_attention_27_gb300 as fa
    inp = make_inputs(1, 2, 2, 333, 128, seed=4)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = nan_forward(q, k, v, causal=True)
    o2, l2 = nan_forward(q, k, v, causal=True, q_offset=0)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.fixture
def tile_rows():
    import exact_attention_27_gb300 as fa
    yield fa.fa_set_forward_tile_rows
    fa.fa_set_forward_tile_rows(0)


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("N,d,causal,Hq,Hkv", [
    (1, 64, True, 2, 1), (129, 64, False, 2, 2), (700, 64, True, 4, 2), (1000, 128, True, 2, 1),
    (257, 128, False, 4, 4), (2048, 64, True, 2, 2), (1, 96, True, 2, 1), (300, 96, False, 4, 2),
    (1000, 96, True, 2, 2), (2048, 96, False, 2, 1),
])
def test_both_tile_sizes_against_the_oracle(tile_rows, rows, N, d, causal, Hq, Hkv):
    """One (128 rows) or two (256) query tiles per CTA, forced, at d = 64, 96 and 128."""
    tile_rows(rows)
    inp = make_inputs(1, Hq, Hkv, N, d, seed=N + d + rows)
    forward_vs_oracle(inp, causal, 1.0 / math.sqrt(d))


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("d", [96, 128])
def test_both_tile_sizes_with_query_offset(tile_rows, rows, d):
    import exact_attention_27_gb300 as fa
    tile_rows(rows)
    inp = make_inputs(1, 4, 2, 300, d, seed=31, Nk=941)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = nan_forward(q, k, v, causal=True, scale=0.1, q_offset=641)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention_forward(as_f64(inp["q"]), as_f64(inp["k"]), as_f64(inp["v"]),
                                            0.1, True, q_offset=641)
    check_forward(o, lse, o_ref, l_ref, f"rows {rows}")


def test_tile_rows_rejects_other_values():
    import exact_attention_27_gb300 as fa
    with pytest.raises(fa.FaError):
        fa.fa_set_forward_tile_rows(64)
    fa.fa_set_forward_tile_rows(0)


@pytest.mark.parametrize("rows_per_cta", [128, 256])
@pytest.mark.parametrize("d", [64, 96, 128, 256])
def test_long_sequence_one_head(tile_rows, rows_per_cta, d):
    """N = 32768, one head: the last query tile visits 256 key tiles (512 at
    d = 256, whose key tiles have 64 rows).  Both tile sizes (d = 256 always
    runs one tile per CTA); tile edges plus seeded rows against the oracle."""
    tile_rows(rows_per_cta)
    N = 32768
    inp = make_inputs(1, 1, 1, N, d, seed=d + rows_per_cta)
    rng = np.random.default_rng(d)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, N - 129, N - 128, N - 1],
                                     rng.integers(0, N, 16)]))
    forward_vs_oracle(inp, True, 1.0 / math.sqrt(d), rows=rows)


@pytest.mark.parametrize("N,causal,Hq,Hkv", [
    (1, True, 2, 1), (129, False, 2, 2), (300, True, 4, 2), (513, True, 2, 2),
    (1000, False, 2, 1), (1024, True, 4, 4), (2048, True, 8, 2), (777, True, 2, 2),
])
def test_cta_pair_forward_against_the_oracle(tile_rows, N, causal, Hq, Hkv):
    """d = 128 on a pair of CTAs (M = 256 products across the two, four query
    tiles per pair): ragged tails, quads with tiles past N, GQA."""
    tile_rows(512)
    inp = make_inputs(1, Hq, Hkv, N, 128, seed=N + 512)
    forward_vs_oracle(inp, causal, 1.0 / math.sqrt(128))


@pytest.mark.parametrize("N,causal", [(1000, True), (2048, False), (4096, True)])
def test_cta_pair_forward_equals_the_two_tile_forward(tile_rows, N, causal):
    """Both kernels form every score and every P V sum in the same order, so
    the pair's outputs equal the two-tile CTA's bit for bit."""
    inp = make_inputs(2, 4, 2, N, 128, seed=N + 5120)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    tile_rows(256)
    o1, l1 = nan_forward(q, k, v, causal=causal)
    tile_rows(512)
    o2, l2 = nan_forward(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [64, 96, 256])
def test_pair_setting_gives_the_two_tile_result_at_other_head_dims(tile_rows, d):
    """The pair of CTAs exists at d = 128 only; elsewhere 512 rows per CTA
    acts as 256 (at d = 256, where only the one-tile kernel exists, both
    settings run it), so the outputs are the same bits."""
    inp = make_inputs(1, 4, 2, 1000, d, seed=9000 + d)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    tile_rows(256)
    o1, l1 = nan_forward(q, k, v, causal=True)
    tile_rows(512)
    o2, l2 = nan_forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_cta_pair_forward_with_query_offset(tile_rows):
    import exact_attention_27_gb300 as fa
    tile_rows(512)
    inp = make_inputs(1, 4, 2, 300, 128, seed=5130, Nk=941)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = nan_forward(q, k, v, causal=True, scale=0.1, q_offset=641)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    o_ref, l_ref = oracle.attention_forward(as_f64(inp["q"]), as_f64(inp["k"]), as_f64(inp["v"]),
                                            0.1, True, q_offset=641)
    check_forward(o, lse, o_ref, l_ref, "pair offset")
