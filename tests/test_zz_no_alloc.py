"""fa_backward_noalloc: the backward pass for callers that cannot allocate
device memory (their memory is reserved by another allocator, or their host
engine forbids allocation when it enqueues work).  It must give the results of
fa_backward, call after call, while its scratch lives in a fixed array inside
the library instead of the memory pool.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test."""

import ctypes
import math

import pytest
import torch

from parity import check_grads
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from exact_attention_27_gb300 import _build
    _build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_27_gb300 as fa
    return fa.library()


def _call(lib, fn, t, B, Hq, Hkv, N, d, scale, causal):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return getattr(lib, fn)(
        t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), t["o"].data_ptr(),
        t["lse"].data_ptr(), t["do"].data_ptr(), t["dq"].data_ptr(), t["dk"].data_ptr(),
        t["dv"].data_ptr(), B, Hq, Hkv, N, d, ctypes.c_float(scale), int(causal), stream)


def _problem(B, Hq, Hkv, N, d, seed, causal):
    import exact_attention_27_gb300 as fa
    inp = make_inputs(B, Hq, Hkv, N, d, seed=seed, with_grad=True)
    t = {n: inp[n].cuda() for n in ("q", "k", "v", "do")}
    t["o"], t["lse"] = fa.attention_forward(t["q"], t["k"], t["v"], causal=causal,
                                            scale=1.0 / math.sqrt(d))
    return t


def _fresh_grads(t):
    # NaN-filled so that any element the call fails to write shows up
    return {"dq": torch.full_like(t["q"], float("nan")),
            "dk": torch.full_like(t["k"], float("nan")),
            "dv": torch.full_like(t["v"], float("nan"))}


@pytest.mark.parametrize("shape", [
    ("causal_train_n4096_d64", None),
    ("gqa_ragged_d128", (1, 4, 2, 777, 128, False)),
])
def test_matches_fa_backward_on_two_calls_in_a_row(lib, shape):
    name, custom = shape
    if custom is None:
        w = WORKLOADS[name]
        B, Hq, Hkv, N, d, causal = w.B, w.Hq, w.Hkv, w.N, w.d, w.causal
    else:
        B, Hq, Hkv, N, d, causal = custom
    scale = 1.0 / math.sqrt(d)
    t = _problem(B, Hq, Hkv, N, d, seed=31, causal=causal)
    ref = dict(t, **_fresh_grads(t))
    assert _call(lib, "fa_backward", ref, B, Hq, Hkv, N, d, scale, causal) == 0
    torch.cuda.synchronize()
    ref_grads = [ref[n].double().cpu().numpy() for n in ("dq", "dk", "dv")]
    for call in range(2):
        out = dict(t, **_fresh_grads(t))
        assert _call(lib, "fa_backward_noalloc", out, B, Hq, Hkv, N, d, scale, causal) == 0
        torch.cuda.synchronize()
        check_grads([out["dq"], out["dk"], out["dv"]], ref_grads, f"no-alloc call {call + 1}")
    import exact_attention_27_gb300 as fa
    assert fa.fa_last_device_error() == 0


def test_rejects_problems_larger_than_its_scratch(lib):
    limit = 32 * 1024 * 1024
    # B*H_q*N*(d+1)*4 bytes just over the limit: rejected before any launch
    N = limit // (65 * 4) + 128
    t = {n: torch.empty(16, dtype=torch.uint8, device="cuda") for n in
         ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv")}
    assert _call(lib, "fa_backward_noalloc", t, 1, 1, 1, N, 64, 0.125, True) == 1
    # a problem that fits is accepted by the same check
    small = _problem(1, 2, 1, 256, 64, seed=5, causal=True)
    small.update(_fresh_grads(small))
    assert _call(lib, "fa_backward_noalloc", small, 1, 2, 1, 256, 64, 0.125, True) == 0
    torch.cuda.synchronize()
