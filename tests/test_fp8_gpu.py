"""FP8 forward parity: fa_forward_fp8 (e4m3 Q, K, V^T with per-tensor descales)
against the oracle's exact attention on the same e4m3 values, decoded exactly
to double and multiplied by their descales.

Tolerance, from the arithmetic of the FP8 path.  Products of e4m3 values are
exact in fp32 and the fp32 accumulation of S adds a negligible error; the
running maximum m_ref of the lazy rescale is at most 8 (log2 units) below
the row maximum, so the kernel's p_j = 2^(s_j c - m_ref) lie in [0, 2^8] and
its running sum is l = 2^(M - m_ref) Z >= Z, with Z = sum_j exp(S_ij - max_i)
in the oracle's terms.  P is rounded to e4m3 for P V: |p~ - p| <= 2^-4 p in
the normal range and <= 2^-10 below it (half the subnormal spacing 2^-9),
with no saturation (2^8 < 448).  The sum l uses the unrounded p.  Hence, per
output element,

    |O_gpu - O_ref| <= v_descale * sum_j (2^-4 P_ij + 2^-10 / Z_i) |v_jc|
                       + 2^-8 |O_ref| + 1e-4,

the 2^-8 term covering the bf16 rounding of O.  L is computed from the fp32
p as in the bf16 path: max abs error 1e-3.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_27_gb300 import _build
    _build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def fp8_inputs(B, Hq, Hkv, N, d, seed, q_ds=1.0, k_ds=1.0, v_ds=1.0):
    """Seeded N(0,1) inputs divided by their descales and rounded to e4m3;
    returns the e4m3 tensors (v transposed) and their exact values in double."""
    inp = make_inputs(B, Hq, Hkv, N, d, seed=seed)
    q8 = (inp["q"].float() / q_ds).to(torch.float8_e4m3fn)
    k8 = (inp["k"].float() / k_ds).to(torch.float8_e4m3fn)
    v8 = (inp["v"].float() / v_ds).to(torch.float8_e4m3fn)
    exact = {"q": q8.to(torch.float64).numpy() * q_ds, "k": k8.to(torch.float64).numpy() * k_ds,
             "v": v8.to(torch.float64).numpy() * v_ds}
    return q8, k8, v8.transpose(-1, -2).contiguous(), exact


def bound(ex, scale, causal, o_ref, v_ds):
    """The per-element error bound of the module docstring, from exact P."""
    q, k, v = ex["q"], ex["k"], ex["v"]
    B, Hq, N, d = q.shape
    G = Hq // k.shape[1]
    out = np.empty_like(o_ref)
    for b in range(B):
        for h in range(Hq):
            s = scale * (q[b, h] @ k[b, h // G].T)
            if causal:
                s[np.triu_indices(N, 1)] = -np.inf
            mx = s.max(axis=1, keepdims=True)
            e = np.exp(s - mx)
            Z = e.sum(axis=1, keepdims=True)
            P = e / Z
            av = np.abs(v[b, h // G]) / v_ds  # |stored v|
            out[b, h] = v_ds * (2.0 ** -4 * (P @ av) + 2.0 ** -10 * (np.where(np.isfinite(s), 1.0, 0.0) @ av) / Z)
    return out + 2.0 ** -8 * np.abs(o_ref) + 1e-4


def run_fp8(q8, k8, vt8, scale, causal, ds):
    import exact_attention_27_gb300 as fa
    q, k, vt = q8.cuda(), k8.cuda(), vt8.cuda()
    # NaN-filled, so that an element the kernel does not write fails the checks.
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_forward_fp8(q, k, vt, o, lse, scale, causal, *ds)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("B,Hq,Hkv,N,causal,ds", [
    (1, 2, 1, 256, False, (1.0, 1.0, 1.0)),
    (1, 2, 1, 256, True, (1.0, 1.0, 1.0)),
    (1, 4, 2, 80, True, (0.5, 2.0, 0.25)),        # ragged: one partial key tile
    (2, 2, 2, 1040, True, (0.125, 0.125, 0.5)),   # ragged tail, descales
    (1, 4, 1, 1024, False, (1.0, 0.5, 2.0)),
    (1, 4, 2, 2048, True, (0.25, 0.25, 0.25)),
])
def test_fp8_forward_within_the_rounding_bound(B, Hq, Hkv, N, causal, ds):
    d = 128
    scale = 1.0 / math.sqrt(d)
    q8, k8, vt8, ex = fp8_inputs(B, Hq, Hkv, N, d, seed=800 + N, q_ds=ds[0], k_ds=ds[1], v_ds=ds[2])
    o, lse = run_fp8(q8, k8, vt8, scale, causal, ds)
    o_ref, l_ref = oracle.attention_forward(ex["q"], ex["k"], ex["v"], scale, causal)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert np.abs(lse - l_ref).max() <= 1e-3
    err = np.abs(o - o_ref)
    bd = bound(ex, scale, causal, o_ref, ds[2])
    worst = np.unravel_index(np.argmax(err - bd), err.shape)
    assert np.all(err <= bd), f"err {err[worst]:.3e} > bound {bd[worst]:.3e} at {worst}"
    # and the typical error is far below the worst case
    assert err.mean() <= 0.25 * bd.mean()


def test_fp8_causal_first_row_is_v0():
    """Query 0 sees key 0 only: P = 1 exactly (e4m3 holds 1), so O[0] is v_0
    times its descale, rounded to bf16."""
    d, ds = 128, (1.0, 1.0, 0.5)
    q8, k8, vt8, ex = fp8_inputs(1, 2, 2, 160, d, seed=5, v_ds=ds[2])
    o, _ = run_fp8(q8, k8, vt8, 1.0 / math.sqrt(d), True, ds)
    want = torch.from_numpy(ex["v"][:, :, 0]).to(torch.bfloat16).double().numpy()
    assert np.array_equal(o[:, :, 0], want)


def test_fp8_forward_ignores_the_tile_rows_setting():
    """The FP8 forward has one kernel (two 128-row query tiles per CTA);
    fa_set_forward_tile_rows leaves its output unchanged, bit for bit."""
    import exact_attention_27_gb300 as fa
    d = 128
    q8, k8, vt8, ex = fp8_inputs(1, 4, 2, 1040, d, seed=8123)  # N a multiple of 16
    outs = []
    try:
        for rows in (0, 128, 256, 512):
            fa.fa_set_forward_tile_rows(rows)
            outs.append(run_fp8(q8, k8, vt8, 1.0 / math.sqrt(d), True, (1.0, 1.0, 1.0)))
    finally:
        fa.fa_set_forward_tile_rows(0)
    for o, lse in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(lse, outs[0][1])
