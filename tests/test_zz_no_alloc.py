"""fa_backward_noalloc: the backward pass for callers that cannot allocate
device memory (their memory is reserved by another allocator, or their host
engine forbids allocation when it enqueues work).  It must give the oracle's
gradients, and those of fa_backward, call after call, while its scratch lives
in a fixed array inside the library instead of the memory pool.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test."""

import ctypes
import math

import pytest
import torch

import oracle
from parity import check_grads, nan_forward, nan_grads
from workloads import WORKLOADS, as_f64, make_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 * 1024 * 1024  # FA_NOALLOC_SCRATCH_BYTES


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


def _scratch_need(B, Hq, N, d):
    """Bytes the call needs: D padded to 1 KiB, then the fp32 dQ accumulator."""
    rows = B * Hq * N
    return -(-rows * 4 // 1024) * 1024 + rows * d * 4


class _Problem:
    """Seeded inputs on the CPU (for the oracle) and on the device, the forward
    outputs, and NaN-filled gradient buffers."""

    def __init__(self, B, Hq, Hkv, N, d, causal, seed):
        self.shape = (B, Hq, Hkv, N, d)
        self.causal = causal
        self.scale = 1.0 / math.sqrt(d)
        self.inp = make_inputs(B, Hq, Hkv, N, d, seed=seed, with_grad=True)
        self.t = {n: self.inp[n].cuda() for n in ("q", "k", "v", "do")}
        self.t["o"], self.t["lse"] = nan_forward(self.t["q"], self.t["k"], self.t["v"],
                                                 causal=causal, scale=self.scale)
        self.new_grads()

    def new_grads(self):
        self.t["dq"], self.t["dk"], self.t["dv"] = nan_grads(self.t["q"], self.t["k"])

    def call(self, lib, fn):
        return _call(lib, fn, self.t, *self.shape, self.scale, self.causal)

    def grads(self):
        return [self.t[n] for n in ("dq", "dk", "dv")]

    def oracle_grads(self):
        f = {n: as_f64(self.inp[n]) for n in ("q", "k", "v", "do")}
        return oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], self.scale,
                                         self.causal)


@pytest.mark.parametrize("shape", [
    ("causal_train_n4096_d64", None),
    ("non-causal GQA ragged d128", (1, 4, 2, 777, 128, False)),
    ("causal GQA d96", (1, 8, 2, 1000, 96, True)),
    ("causal GQA d256", (1, 8, 2, 1000, 256, True)),
])
def test_matches_the_oracle_and_fa_backward_on_two_calls_in_a_row(lib, shape):
    name, custom = shape
    if custom is None:
        w = WORKLOADS[name]
        B, Hq, Hkv, N, d, causal = w.B, w.Hq, w.Hkv, w.N, w.d, w.causal
    else:
        B, Hq, Hkv, N, d, causal = custom
    pr = _Problem(B, Hq, Hkv, N, d, causal, seed=31)
    ref_oracle = pr.oracle_grads()
    assert pr.call(lib, "fa_backward") == 0
    torch.cuda.synchronize()
    ref_gpu = [g.double().cpu().numpy() for g in pr.grads()]
    check_grads(pr.grads(), ref_oracle, f"{name}: fa_backward")
    for call in range(2):
        pr.new_grads()
        assert pr.call(lib, "fa_backward_noalloc") == 0
        torch.cuda.synchronize()
        check_grads(pr.grads(), ref_oracle, f"{name}: no-alloc call {call + 1} vs the oracle")
        check_grads(pr.grads(), ref_gpu, f"{name}: no-alloc call {call + 1} vs fa_backward")
    import exact_attention_27_gb300 as fa
    assert fa.fa_last_device_error() == 0


def test_back_to_back_calls_on_one_stream(lib):
    """Two calls with different inputs and the same shapes enqueued one after
    the other with no synchronisation between them (the second reuses the
    shared scratch while the first may still be finishing), then fa_forward,
    fa_backward_noalloc and fa_backward interleaved on the same stream.  Every
    call's gradients against the oracle."""
    B, Hq, Hkv, N, d, causal = 2, 8, 4, 1500, 64, True
    a = _Problem(B, Hq, Hkv, N, d, causal, seed=101)
    b = _Problem(B, Hq, Hkv, N, d, causal, seed=202)
    torch.cuda.synchronize()
    assert a.call(lib, "fa_backward_noalloc") == 0
    assert b.call(lib, "fa_backward_noalloc") == 0
    torch.cuda.synchronize()
    ref_a, ref_b = a.oracle_grads(), b.oracle_grads()
    check_grads(a.grads(), ref_a, "first of two back-to-back calls")
    check_grads(b.grads(), ref_b, "second of two back-to-back calls")

    import exact_attention_27_gb300 as fa
    c = _Problem(B, Hq, Hkv, N, d, causal, seed=303)
    ref_c = c.oracle_grads()
    a.new_grads()
    b.new_grads()
    c.new_grads()
    torch.cuda.synchronize()
    # forward of c, no-alloc backward of a, pooled backward of b, no-alloc of c
    c.t["o"].fill_(float("nan"))
    fa.fa_forward(c.t["q"], c.t["k"], c.t["v"], c.t["o"], c.t["lse"], c.scale, causal)
    assert a.call(lib, "fa_backward_noalloc") == 0
    assert b.call(lib, "fa_backward") == 0
    assert c.call(lib, "fa_backward_noalloc") == 0
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    check_grads(a.grads(), ref_a, "interleaved: no-alloc after a forward")
    check_grads(b.grads(), ref_b, "interleaved: fa_backward between two no-alloc calls")
    check_grads(c.grads(), ref_c, "interleaved: no-alloc on the interleaved forward's output")


def test_problem_that_exactly_fills_the_scratch(lib):
    """B*H_q*N = 129052 rows at d = 64 need exactly the scratch's size
    (505 KiB of D + 129052*64*4 bytes of accumulator = 32 MiB): accepted and
    correct against the oracle (causal, four query heads per K/V head).  One
    more position per head is rejected before anything is launched."""
    B, Hq, Hkv, N, d = 1, 28, 7, 4609, 64
    assert _scratch_need(B, Hq, N, d) == SCRATCH_BYTES
    pr = _Problem(B, Hq, Hkv, N, d, True, seed=17)
    assert pr.call(lib, "fa_backward_noalloc") == 0
    torch.cuda.synchronize()
    check_grads(pr.grads(), pr.oracle_grads(), "exactly full scratch")
    assert _scratch_need(B, Hq, N + 1, d) > SCRATCH_BYTES
    big = _Problem(B, Hq, Hkv, N + 1, d, True, seed=18)
    assert big.call(lib, "fa_backward_noalloc") == 1  # FA_ERR_INVALID_ARGUMENT
    torch.cuda.synchronize()
    assert torch.isnan(big.t["dq"]).all()  # nothing was launched


def test_rejects_problems_larger_than_its_scratch(lib):
    # B*H_q*N*(d+1)*4 bytes just over the limit: rejected before any launch
    N = SCRATCH_BYTES // (65 * 4) + 128
    t = {n: torch.empty(16, dtype=torch.uint8, device="cuda") for n in
         ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv")}
    assert _call(lib, "fa_backward_noalloc", t, 1, 1, 1, N, 64, 0.125, True) == 1


def _cudart():
    # libfa.so links the shared CUDA runtime, so this finds the loaded copy.
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    pytest.skip("CUDA runtime library not found by name")


def test_allocates_nothing_from_the_memory_pool(lib):
    """The device's current memory pool (where fa_backward's cudaMallocAsync
    draws from) keeps a high-water mark of the bytes in use.  Reset it, run
    the no-allocation call, and it stays at zero; fa_backward, the positive
    control, raises it by at least its scratch."""
    rt = _cudart()
    pool = ctypes.c_void_p()
    dev = torch.cuda.current_device()
    assert rt.cudaDeviceGetMemPool(ctypes.byref(pool), dev) == 0
    USED_HIGH, USED_CURRENT = 8, 7  # cudaMemPoolAttrUsedMemHigh / UsedMemCurrent

    def attr(which):
        v = ctypes.c_uint64(0)
        assert rt.cudaMemPoolGetAttribute(pool, which, ctypes.byref(v)) == 0
        return v.value

    def reset_high():
        zero = ctypes.c_uint64(0)
        assert rt.cudaMemPoolSetAttribute(pool, USED_HIGH, ctypes.byref(zero)) == 0

    B, Hq, Hkv, N, d = 2, 8, 8, 2048, 64
    pr = _Problem(B, Hq, Hkv, N, d, True, seed=55)
    torch.cuda.synchronize()
    reset_high()
    base = attr(USED_HIGH)  # what other users of the pool hold now (normally 0)
    for _ in range(2):
        assert pr.call(lib, "fa_backward_noalloc") == 0
    torch.cuda.synchronize()
    assert attr(USED_HIGH) == base
    reset_high()
    base = attr(USED_HIGH)
    assert pr.call(lib, "fa_backward") == 0
    torch.cuda.synchronize()
    assert attr(USED_HIGH) >= base + _scratch_need(B, Hq, N, d)
    assert attr(USED_CURRENT) <= base  # fa_backward gave its scratch back
