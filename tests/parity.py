"""Helpers shared by the GPU parity tests: tolerances, device runs through the
C-ABI binding, and comparisons against the CPU oracle.

Tolerances (bf16 inputs, fp32 accumulation, bf16 outputs):
  O       max |err| <= 2e-2 and mean |err| <= 2e-3
  L       max |err| <= 1e-3
  dQ/dK/dV  max |err| <= 5e-2 * max |reference|   (per tensor), and never
           below 1e-4: where the exact gradient vanishes (one visible key, so
           the softmax is constant) the relative bound would demand exact zeros,
           while D = rowsum(dO o O) from the bf16 output and dP from the MMA
           differ by fp32 rounding (about d * 2^-24 * |dO| |V|).
"""

import numpy as np
import torch

import oracle
from workloads import as_f64

O_MAX = 2e-2
O_MEAN = 2e-3
L_MAX = 1e-3
GRAD_REL = 5e-2
GRAD_ABS_FLOOR = 1e-4


def gpu_forward(inp, causal, scale):
    import exact_attention_27_gb300 as fa
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.attention_forward(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    return o, lse


def check_forward(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.cpu().numpy().astype(np.float64)
    err = np.abs(o - o_ref)
    lerr = np.abs(lse - lse_ref)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    assert err.max() <= O_MAX, f"{what}: O max err {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{what}: O mean err {err.mean():.3e}"
    assert lerr.max() <= L_MAX, f"{what}: L max err {lerr.max():.3e}"
    return err.max(), err.mean(), lerr.max()


def forward_vs_oracle(inp, causal, scale, rows=None):
    """Runs the GPU forward on `inp` and compares with the oracle (all rows or `rows`)."""
    o, lse = gpu_forward(inp, causal, scale)
    o_ref, l_ref = oracle.attention_forward(as_f64(inp["q"]), as_f64(inp["k"]), as_f64(inp["v"]),
                                            scale, causal, rows=rows)
    if rows is not None:
        o, lse = o[:, :, rows], lse[:, :, rows]
    return check_forward(o, lse, o_ref, l_ref), (o, lse)


def check_grads(got, ref, what=""):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g = g.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all(), f"{what}: {name} not finite"
        bound = max(GRAD_REL * np.abs(r).max(), GRAD_ABS_FLOOR)
        err = np.abs(g - r).max()
        assert err <= bound, f"{what}: {name} max err {err:.3e} > {bound:.3e}"
