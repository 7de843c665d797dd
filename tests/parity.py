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

import concurrent.futures
import os

import numpy as np
import torch

import oracle
from workloads import as_f64

O_MAX = 2e-2
O_MEAN = 2e-3
L_MAX = 1e-3
GRAD_REL = 5e-2
GRAD_ABS_FLOOR = 1e-4


def nan_outputs(q):
    """O and L buffers for a forward on q, filled with NaN so that any element
    the kernels fail to write (or a stale block the allocator hands back)
    shows up in the comparison."""
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device=q.device)
    return o, lse


def nan_grads(q, k):
    """dq, dk, dv buffers filled with NaN (same purpose as nan_outputs)."""
    return (torch.full_like(q, float("nan")), torch.full_like(k, float("nan")),
            torch.full_like(k, float("nan")))


def nan_forward(q, k, v, causal=False, scale=None, q_offset=None):
    """The binding's attention_forward (fa_forward, or fa_forward_ex for a
    query offset or unequal lengths) into NaN-filled outputs."""
    import math

    import exact_attention_27_gb300 as fa
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    o, lse = nan_outputs(q)
    if q_offset is None and q.shape[2] == k.shape[2]:
        fa.fa_forward(q, k, v, o, lse, scale, causal)
    else:
        fa.fa_forward_ex(q, k, v, o, lse, scale, causal, q_offset or 0)
    return o, lse


def nan_backward(q, k, v, o, lse, do, causal=False, scale=None, deterministic=False):
    """The binding's attention_backward into NaN-filled gradient buffers."""
    import math

    import exact_attention_27_gb300 as fa
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    dq, dk, dv = nan_grads(q, k)
    run = fa.fa_backward_deterministic if deterministic else fa.fa_backward
    run(q, k, v, o, lse, do, dq, dk, dv, scale, causal)
    return dq, dk, dv


def gpu_forward(inp, causal, scale):
    """fa_forward on the inputs of `inp` (CPU tensors) into NaN-filled outputs."""
    import exact_attention_27_gb300 as fa
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = nan_outputs(q)
    fa.fa_forward(q, k, v, o, lse, scale, causal)
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


def forward_every_element(inp, causal, scale, o_gpu, lse_gpu, block_rows=512, what=""):
    """Compares every element of a GPU forward with the oracle, evaluating the
    oracle on blocks of `block_rows` query rows (all heads at once) so that the
    host memory it holds for S and P stays bounded at full size.  The error
    statistics are those of check_forward over the whole output."""
    o_all = o_gpu.float().cpu()
    l_all = lse_gpu.cpu()
    assert torch.isfinite(o_all).all() and torch.isfinite(l_all).all(), what
    qf, kf, vf = (as_f64(inp[n]) for n in ("q", "k", "v"))
    B, H, N = qf.shape[:3]

    def block(r0):
        r1 = min(N, r0 + block_rows)
        o_ref, l_ref = oracle.attention_forward(qf, kf, vf, scale, causal,
                                                rows=np.arange(r0, r1))
        err = np.abs(o_all[:, :, r0:r1].numpy().astype(np.float64) - o_ref)
        lerr = np.abs(l_all[:, :, r0:r1].numpy().astype(np.float64) - l_ref)
        return float(err.max()), float(err.sum()), float(lerr.max())

    # The oracle runs its heads in parallel; with fewer heads than host cores,
    # row blocks run concurrently too (the C call releases the interpreter).
    workers = max(1, (os.cpu_count() or 1) // (B * H))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        parts = list(ex.map(block, range(0, N, block_rows)))
    o_max = max(x[0] for x in parts)
    o_sum = sum(x[1] for x in parts)
    l_max = max(x[2] for x in parts)
    o_mean = o_sum / o_all.numel()
    assert o_max <= O_MAX, f"{what}: O max err {o_max:.3e}"
    assert o_mean <= O_MEAN, f"{what}: O mean err {o_mean:.3e}"
    assert l_max <= L_MAX, f"{what}: L max err {l_max:.3e}"
    return o_max, o_mean, l_max
