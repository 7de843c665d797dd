"""Exact attention oracle (double precision, CPU).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline / reference leg may import this package.  The CUDA library never
links, loads or calls it, and it never imports the CUDA library.

`fa_oracle.c` states the plain definition (S and P materialised, see its
header for the passages it follows); this module builds it with gcc, loads it
with ctypes and wraps it for numpy arrays.  `online_softmax` holds the pages'
blockwise update rules for a single row, used to check the worked examples.
"""

import ctypes
import os
import subprocess
import threading

import numpy as np

from .online_softmax import naive_block_average, online_softmax_row  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(src=_SRC, out=_LIB, extra_flags=()):
    """Compile `src` into the shared library `out` with gcc (OpenMP if present)."""
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", src, "-o", out, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + list(extra_flags),
                       check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + list(extra_flags), check=True, capture_output=True)
    return out


def _declare(lib):
    i64, dbl, p = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    lib.oracle_attention_forward.restype = ctypes.c_int
    lib.oracle_attention_forward.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i64,
                                             dbl, ctypes.c_int, i64, p, i64]
    lib.oracle_attention_backward.restype = ctypes.c_int
    lib.oracle_attention_backward.argtypes = [p, p, p, p, p, p, p, p, i64, i64, i64, i64, i64,
                                              i64, dbl, ctypes.c_int, i64]
    lib.oracle_row_dot.restype = ctypes.c_int
    lib.oracle_row_dot.argtypes = [p, p, p, i64, i64]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    return lib


def load(path=None):
    """Load an oracle library: the default one (built on first use) or `path`."""
    global _lib
    if path is not None:
        return Oracle(_declare(ctypes.CDLL(path)))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB)
                    or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
                build()
            _lib = Oracle(_declare(ctypes.CDLL(_LIB)))
    return _lib


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape:
        raise ValueError("expected q [B,Hq,Nq,d] and k, v [B,Hkv,Nk,d] of equal shape")
    if q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError("q and k/v differ in batch or head dimension")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """numpy front end to one loaded copy of the C oracle."""

    def __init__(self, lib):
        self.lib = lib

    def num_threads(self):
        return int(self.lib.oracle_num_threads())

    def forward(self, q, k, v, scale, causal, q_offset=0, rows=None):
        """O and L for q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d] (any float dtype).

        Returns (o, lse) as float64: o [B,Hq,R,d], lse [B,Hq,R] where R = Nq,
        or len(rows) when `rows` selects query rows (same rows in every head).
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        _check_shapes(q, k, v)
        B, Hq, Nq, d = q.shape
        _, Hkv, Nk, _ = k.shape
        if rows is None:
            rr, R, rp = None, Nq, None
        else:
            rr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
            R, rp = rr.shape[0], _ptr(rr)
        o = np.zeros((B, Hq, R, d))
        lse = np.zeros((B, Hq, R))
        rc = self.lib.oracle_attention_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                               B, Hq, Hkv, Nq, Nk, d, float(scale), int(causal),
                                               int(q_offset), rp, R)
        if rc != 0:
            raise RuntimeError(f"oracle_attention_forward failed with code {rc}")
        return o, lse

    def backward(self, q, k, v, dout, scale, causal, q_offset=0, want_rowdot=False):
        """(dq, dk, dv[, rowdot]) as float64 for the same shapes as `forward`."""
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        _check_shapes(q, k, v)
        if dout.shape != q.shape:
            raise ValueError("dout must have q's shape")
        B, Hq, Nq, d = q.shape
        _, Hkv, Nk, _ = k.shape
        dq = np.zeros_like(q)
        dk = np.zeros_like(k)
        dv = np.zeros_like(v)
        rowdot = np.zeros((B, Hq, Nq)) if want_rowdot else None
        rc = self.lib.oracle_attention_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq),
                                                _ptr(dk), _ptr(dv),
                                                _ptr(rowdot) if want_rowdot else None,
                                                B, Hq, Hkv, Nq, Nk, d, float(scale), int(causal),
                                                int(q_offset))
        if rc != 0:
            raise RuntimeError(f"oracle_attention_backward failed with code {rc}")
        return (dq, dk, dv, rowdot) if want_rowdot else (dq, dk, dv)


    def row_dot(self, a, b):
        """sum over the last axis of a * b, for arrays of equal shape [..., d]."""
        a, b = _f64(a), _f64(b)
        if a.shape != b.shape or a.ndim < 1:
            raise ValueError("row_dot needs two arrays of equal shape")
        out = np.zeros(a.shape[:-1])
        rc = self.lib.oracle_row_dot(_ptr(a), _ptr(b), _ptr(out), a.size // a.shape[-1],
                                     a.shape[-1])
        if rc != 0:
            raise RuntimeError(f"oracle_row_dot failed with code {rc}")
        return out


def row_dot(a, b):
    return load().row_dot(a, b)


def attention_forward(q, k, v, scale, causal, q_offset=0, rows=None):
    return load().forward(q, k, v, scale, causal, q_offset, rows)


def attention_backward(q, k, v, dout, scale, causal, q_offset=0, want_rowdot=False):
    return load().backward(q, k, v, dout, scale, causal, q_offset, want_rowdot)


def num_threads():
    return load().num_threads()
