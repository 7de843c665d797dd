"""The C-ABI library loads, exports every function include/fa.h declares, and
rejects invalid arguments on the host before any CUDA call (no GPU needed)."""

import ctypes
import os
import re

import pytest

import exact_attention_27_gb300 as fa
from exact_attention_27_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fa_forward", "fa_backward", "fa_status_string", "fa_last_device_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(5):
        s = fa.fa_status_string(code)
        assert isinstance(s, str) and s
    assert fa.fa_status_string(0) == "ok"


# Fake, 16-byte aligned, never dereferenced: validation fails before any use.
P = ctypes.c_void_p(0x10000)
Q = ctypes.c_void_p(0x10008)  # 8-byte aligned only


def fwd(lib, q=P, k=P, v=P, o=P, lse=P, B=1, Hq=2, Hkv=1, N=64, d=64, scale=0.125, causal=0):
    return lib.fa_forward(q, k, v, o, lse, B, Hq, Hkv, N, d, ctypes.c_float(scale), causal, None)


def bwd(lib, d=64, **kw):
    args = dict(q=P, k=P, v=P, o=P, lse=P, do=P, dq=P, dk=P, dv=P, B=1, Hq=2, Hkv=1, N=64,
                scale=0.125, causal=1)
    args.update(kw)
    return lib.fa_backward(args["q"], args["k"], args["v"], args["o"], args["lse"], args["do"],
                           args["dq"], args["dk"], args["dv"], args["B"], args["Hq"], args["Hkv"],
                           args["N"], d, ctypes.c_float(args["scale"]), args["causal"], None)


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(lse=None), dict(B=0), dict(N=0), dict(Hq=3, Hkv=2), dict(Hkv=0),
    dict(scale=0.0), dict(scale=-1.0), dict(scale=float("nan")), dict(scale=float("inf")),
    dict(causal=2), dict(q=Q), dict(o=Q), dict(N=65536 * 128 + 1),
])
def test_forward_rejects_invalid_arguments(lib, kw):
    assert fwd(lib, **kw) == fa.FA_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("d", [0, 32, 80, 160, 192, 512])
def test_forward_rejects_unsupported_head_dim(lib, d):
    assert fwd(lib, d=d) == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw", [dict(do=None), dict(dq=None), dict(dk=Q), dict(Hq=3, Hkv=2),
                                dict(scale=0.0), dict(N=-5)])
def test_backward_rejects_invalid_arguments(lib, kw):
    assert bwd(lib, **kw) == fa.FA_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("d", [0, 32, 80, 160, 192, 512])
def test_backward_rejects_unsupported_head_dim(lib, d):
    assert bwd(lib, d=d) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_backward_deterministic(P, P, P, P, P, P, P, P, P, 1, 2, 1, 64, d,
                                         ctypes.c_float(0.125), 1, None) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_backward_noalloc(P, P, P, P, P, P, P, P, P, 1, 2, 1, 64, d,
                                   ctypes.c_float(0.125), 1, None) == fa.FA_ERR_UNSUPPORTED


def test_preprocess_rejects_invalid_arguments(lib):
    assert lib.fa_backward_preprocess(P, P, P, 0, 64, None) == fa.FA_ERR_INVALID_ARGUMENT
    assert lib.fa_backward_preprocess(None, P, P, 4, 64, None) == fa.FA_ERR_INVALID_ARGUMENT
    assert lib.fa_backward_preprocess(Q, P, P, 4, 64, None) == fa.FA_ERR_INVALID_ARGUMENT
    assert lib.fa_backward_preprocess(P, P, P, 4, 48, None) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_backward_preprocess(P, P, P, 4, 512, None) == fa.FA_ERR_UNSUPPORTED


def test_selftest_rejects_out_of_range_limit(lib):
    assert lib.fa_selftest_wait_timeout(0, None) == fa.FA_ERR_INVALID_ARGUMENT
    assert lib.fa_selftest_wait_timeout(5000, None) == fa.FA_ERR_INVALID_ARGUMENT


def test_binding_checks_tensors_before_the_library():
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)  # CPU tensor
    with pytest.raises(ValueError):
        fa.fa_forward(q, q, q, q, torch.zeros(1, 1, 8), 0.125, False)


def test_product_path_never_touches_the_oracle():
    """The package and its CUDA sources never name the oracle."""
    pkg = os.path.join(ROOT, "exact_attention_27_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f


def fwd_ex(lib, Nq=16, Nk=64, off=48, d=64, causal=1, q=P):
    return lib.fa_forward_ex(q, P, P, P, P, 1, 2, 1, Nq, Nk, d, ctypes.c_float(0.125), causal,
                             off, None)


@pytest.mark.parametrize("kw", [dict(off=-1), dict(Nk=0), dict(Nq=0), dict(q=Q), dict(causal=3),
                                dict(off=2**31 - 10)])
def test_forward_ex_rejects_invalid_arguments(lib, kw):
    assert fwd_ex(lib, **kw) == fa.FA_ERR_INVALID_ARGUMENT


def test_forward_ex_rejects_unsupported_head_dim(lib):
    assert fwd_ex(lib, d=32) == fa.FA_ERR_UNSUPPORTED


def fwd_fp8(lib, d=128, N=64, q=P, vt=P, qd=1.0, kd=1.0, vd=1.0, causal=1):
    return lib.fa_forward_fp8(q, P, vt, P, P, 1, 2, 1, N, d, ctypes.c_float(0.125),
                              ctypes.c_float(qd), ctypes.c_float(kd), ctypes.c_float(vd), causal,
                              None)


@pytest.mark.parametrize("kw", [dict(N=72), dict(N=1), dict(qd=0.0), dict(kd=-1.0),
                                dict(vd=float("nan")), dict(vd=float("inf")), dict(q=None),
                                dict(vt=Q), dict(causal=2), dict(qd=1e30, kd=1e30)])
def test_forward_fp8_rejects_invalid_arguments(lib, kw):
    assert fwd_fp8(lib, **kw) == fa.FA_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("d", [64, 96, 256])
def test_forward_fp8_rejects_unsupported_head_dim(lib, d):
    assert fwd_fp8(lib, d=d) == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("rows", [-1, 1, 64, 127, 384, 1024])
def test_forward_tile_rows_rejects_other_values(lib, rows):
    assert lib.fa_set_forward_tile_rows(rows) == fa.FA_ERR_INVALID_ARGUMENT
    assert lib.fa_set_forward_tile_rows(0) == fa.FA_OK
