"""Exact attention on NVIDIA GB300: Python binding of the C-ABI library.

The functions here carry the names of the C entry points in include/fa.h and
only marshal arguments: they check dtypes and shapes of PyTorch tensors, pass
their device pointers and the current CUDA stream to libfa.so, and turn a
non-zero status into `FaError`.  Every step of the computation runs in the
library's CUDA kernels; there is no other implementation behind these calls.
If libfa.so is missing or cannot be loaded, importing the binding succeeds but
every call raises.

    o, lse = attention_forward(q, k, v, causal=True)
    dq, dk, dv = attention_backward(q, k, v, o, lse, do, causal=True)
"""

import ctypes
import math

from ._lib import FaError, library, status_string  # noqa: F401

__all__ = [
    "FaError", "fa_forward", "fa_forward_ex", "fa_forward_fp8", "fa_set_forward_tile_rows", "fa_forward_tile_rows_for",
    "fa_backward", "fa_backward_deterministic", "fa_backward_preprocess", "fa_status_string",
    "fa_last_device_error", "fa_selftest_wait_timeout", "fa_set_backward_events", "attention_forward", "attention_backward",
    "library",
]

FA_OK = 0
FA_ERR_INVALID_ARGUMENT = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_DEVICE_TIMEOUT = 4


# torch is imported on first use; the current-stream handle is read with
# torch's raw getter where it has one (a Stream object per call costs
# microseconds of host time).
_torch = None
_BF16 = _F32 = None
_current_stream = None


def _torch_mod():
    global _torch, _BF16, _F32, _current_stream
    if _torch is None:
        import torch
        _BF16, _F32 = torch.bfloat16, torch.float32
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        dev = getattr(torch._C, "_cuda_getDevice", None)
        if raw is not None and dev is not None:
            _current_stream = lambda: raw(dev())
        else:
            _current_stream = lambda: torch.cuda.current_stream().cuda_stream
        _torch = torch
    return _torch


def _stream(stream):
    if stream is None:
        if _torch is None:
            _torch_mod()
        return ctypes.c_void_p(_current_stream())
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, what):
    if status != FA_OK:
        raise FaError(status, what)


def _bf16_cuda(name, t, shape=None):
    if _torch is None:
        _torch_mod()
    if t.dtype is not _BF16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if shape is not None and t.shape != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _f32_cuda(name, t, shape):
    if _torch is None:
        _torch_mod()
    if t.dtype is not _F32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor")
    if t.shape != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _shapes(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be [B, H, N, d]")
    B, Hq, N, d = q.shape
    if k.shape[0] != B or k.shape[2] != N or k.shape[3] != d:
        raise ValueError("k must be [B, H_kv, N, d] with q's B, N and d")
    return B, Hq, k.shape[1], N, d


def fa_forward(q, k, v, o, lse, scale, causal, stream=None):
    """fa_forward of include/fa.h on torch tensors; writes o and lse."""
    B, Hq, Hkv, N, d = _shapes(q, k)
    _bf16_cuda("q", q)
    _bf16_cuda("k", k)
    _bf16_cuda("v", v, k.shape)
    _bf16_cuda("o", o, q.shape)
    _f32_cuda("lse", lse, (B, Hq, N))
    _check(library().fa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), B, Hq, Hkv, N, d, ctypes.c_float(scale),
                                int(bool(causal)), _stream(stream)), "fa_forward")


def fa_forward_ex(q, k, v, o, lse, scale, causal, q_offset=0, stream=None):
    """fa_forward_ex of include/fa.h: q [B,H_q,N_q,d] against k/v [B,H_kv,N_kv,d]."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be [B, H, N, d]")
    B, Hq, Nq, d = q.shape
    if k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k must be [B, H_kv, N_kv, d] with q's B and d")
    Hkv, Nk = k.shape[1], k.shape[2]
    _bf16_cuda("q", q)
    _bf16_cuda("k", k)
    _bf16_cuda("v", v, k.shape)
    _bf16_cuda("o", o, q.shape)
    _f32_cuda("lse", lse, (B, Hq, Nq))
    _check(library().fa_forward_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, Hq, Hkv, Nq, Nk, d, ctypes.c_float(scale),
                                   int(bool(causal)), int(q_offset), _stream(stream)),
           "fa_forward_ex")


def fa_forward_fp8(q, k, v_t, o, lse, scale, causal, q_descale=1.0, k_descale=1.0,
                   v_descale=1.0, stream=None):
    """fa_forward_fp8 of include/fa.h: q [B,H_q,N,d], k [B,H_kv,N,d] and the
    transposed v_t [B,H_kv,d,N] as float8_e4m3fn tensors (values times their
    descales); writes o (bf16) and lse (fp32)."""
    import torch
    B, Hq, Hkv, N, d = _shapes(q, k)
    for name, t, shp in (("q", q, None), ("k", k, None), ("v_t", v_t, (B, Hkv, d, N))):
        if t.dtype != torch.float8_e4m3fn or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float8_e4m3fn CUDA tensor")
        if shp is not None and tuple(t.shape) != tuple(shp):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shp)}")
    _bf16_cuda("o", o, q.shape)
    _f32_cuda("lse", lse, (B, Hq, N))
    _check(library().fa_forward_fp8(q.data_ptr(), k.data_ptr(), v_t.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), B, Hq, Hkv, N, d, ctypes.c_float(scale),
                                    ctypes.c_float(q_descale), ctypes.c_float(k_descale),
                                    ctypes.c_float(v_descale), int(bool(causal)),
                                    _stream(stream)), "fa_forward_fp8")


def fa_set_forward_tile_rows(rows):
    """fa_set_forward_tile_rows of include/fa.h: 0 (per shape), 128, 256 or 512."""
    _check(library().fa_set_forward_tile_rows(int(rows)), "fa_set_forward_tile_rows")


def fa_forward_tile_rows_for(B, H_q, H_kv, N_q, N_kv, d, causal, q_offset, sms):
    """fa_forward_tile_rows_for of include/fa.h: 128 or 256, 0 for invalid sizes."""
    return int(library().fa_forward_tile_rows_for(int(B), int(H_q), int(H_kv), int(N_q),
                                                  int(N_kv), int(d), int(bool(causal)),
                                                  int(q_offset), int(sms)))


def fa_backward(q, k, v, o, lse, do, dq, dk, dv, scale, causal, stream=None):
    """fa_backward of include/fa.h on torch tensors; writes dq, dk, dv."""
    B, Hq, Hkv, N, d = _shapes(q, k)
    for name, t, shp in (("q", q, None), ("k", k, None), ("v", v, k.shape), ("o", o, q.shape),
                         ("do", do, q.shape), ("dq", dq, q.shape), ("dk", dk, k.shape),
                         ("dv", dv, k.shape)):
        _bf16_cuda(name, t, shp)
    _f32_cuda("lse", lse, (B, Hq, N))
    _check(library().fa_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                 dv.data_ptr(), B, Hq, Hkv, N, d, ctypes.c_float(scale),
                                 int(bool(causal)), _stream(stream)), "fa_backward")


def fa_backward_deterministic(q, k, v, o, lse, do, dq, dk, dv, scale, causal, stream=None):
    """fa_backward_deterministic of include/fa.h: bit-reproducible gradients."""
    B, Hq, Hkv, N, d = _shapes(q, k)
    for name, t, shp in (("q", q, None), ("k", k, None), ("v", v, k.shape), ("o", o, q.shape),
                         ("do", do, q.shape), ("dq", dq, q.shape), ("dk", dk, k.shape),
                         ("dv", dv, k.shape)):
        _bf16_cuda(name, t, shp)
    _f32_cuda("lse", lse, (B, Hq, N))
    _check(library().fa_backward_deterministic(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, N, d, ctypes.c_float(scale),
        int(bool(causal)), _stream(stream)), "fa_backward_deterministic")


def fa_backward_preprocess(o, do, D, stream=None):
    """fa_backward_preprocess of include/fa.h: D[r] = sum_c dO[r, c] O[r, c]."""
    _bf16_cuda("o", o)
    _bf16_cuda("do", do, o.shape)
    d = o.shape[-1]
    rows = o.numel() // d
    _f32_cuda("D", D, tuple(o.shape[:-1]))
    _check(library().fa_backward_preprocess(o.data_ptr(), do.data_ptr(), D.data_ptr(), rows, d,
                                            _stream(stream)), "fa_backward_preprocess")


def fa_status_string(status):
    return status_string(status)


def fa_last_device_error(stream=None):
    """Synchronises the stream; returns the status code (0 = FA_OK)."""
    return int(library().fa_last_device_error(_stream(stream)))


def fa_selftest_wait_timeout(limit_ms, stream=None):
    _check(library().fa_selftest_wait_timeout(int(limit_ms), _stream(stream)),
           "fa_selftest_wait_timeout")


def fa_set_backward_events(before, after):
    """Records torch.cuda.Event `before`/`after` around the backward main kernel
    of later fa_backward calls (None, None switches the hook off)."""
    h = (lambda e: ctypes.c_void_p(e.cuda_event) if e is not None else None)
    library().fa_set_backward_events(h(before), h(after))


def attention_forward(q, k, v, causal=False, scale=None, q_offset=None, stream=None):
    """Allocates o and lse on q's device and runs fa_forward (or fa_forward_ex
    when q and k differ in length or a query offset is given); returns (o, lse)."""
    import torch
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    if q_offset is None and q.shape[2] == k.shape[2]:
        fa_forward(q, k, v, o, lse, scale, causal, stream)
    else:
        fa_forward_ex(q, k, v, o, lse, scale, causal, q_offset or 0, stream)
    return o, lse


def attention_backward(q, k, v, o, lse, do, causal=False, scale=None, deterministic=False,
                       stream=None):
    """Allocates dq, dk, dv on q's device and runs fa_backward (or
    fa_backward_deterministic); returns them."""
    import torch
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    run = fa_backward_deterministic if deterministic else fa_backward
    run(q, k, v, o, lse, do, dq, dk, dv, scale, causal, stream)
    return dq, dk, dv
