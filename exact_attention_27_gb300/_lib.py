"""Loads libfa.so (built in-tree by `_build.py`) and declares its C signatures."""

import ctypes
import os
import threading

from ._build import LIB_PATH

_lock = threading.Lock()
_lib = None
_load_error = None

_STATUS = {
    0: "ok",
    1: "invalid argument",
    2: "unsupported head dimension",
    3: "CUDA runtime error",
    4: "a bounded wait inside a kernel ran out",
}


class FaError(RuntimeError):
    """A non-zero fa_status returned by the CUDA library."""

    def __init__(self, status, what=""):
        self.status = int(status)
        super().__init__(f"{what}: {status_string(self.status)} (status {self.status})")


def status_string(status):
    if _lib is not None:
        return _lib.fa_status_string(int(status)).decode()
    return _STATUS.get(int(status), "unknown status")


def _declare(lib):
    p, i, f, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong
    lib.fa_forward.restype = i
    lib.fa_forward.argtypes = [p, p, p, p, p, i, i, i, i, i, f, i, p]
    lib.fa_forward_ex.restype = i
    lib.fa_forward_ex.argtypes = [p, p, p, p, p, i, i, i, i, i, i, f, i, i, p]
    lib.fa_forward_fp8.restype = i
    lib.fa_set_forward_tile_rows.restype = i
    lib.fa_set_forward_tile_rows.argtypes = [i]
    lib.fa_forward_fp8.argtypes = [p, p, p, p, p, i, i, i, i, i, f, f, f, f, i, p]
    lib.fa_backward.restype = i
    lib.fa_backward.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, f, i, p]
    lib.fa_backward_deterministic.restype = i
    lib.fa_backward_deterministic.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, f, i, p]
    lib.fa_backward_noalloc.restype = i
    lib.fa_backward_noalloc.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, f, i, p]
    lib.fa_backward_preprocess.restype = i
    lib.fa_backward_preprocess.argtypes = [p, p, p, ll, i, p]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_status_string.argtypes = [i]
    lib.fa_last_device_error.restype = i
    lib.fa_last_device_error.argtypes = [p]
    lib.fa_set_backward_events.restype = None
    lib.fa_set_backward_events.argtypes = [p, p]
    lib.fa_selftest_wait_timeout.restype = i
    lib.fa_selftest_wait_timeout.argtypes = [i, p]
    return lib


def library():
    """The loaded CUDA library; raises if it was not built or cannot load."""
    global _lib, _load_error
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None and _load_error is None:
            if not os.path.exists(LIB_PATH):
                _load_error = (f"{LIB_PATH} is missing: build it with "
                               "`python -m exact_attention_27_gb300._build`")
            else:
                try:
                    _lib = _declare(ctypes.CDLL(LIB_PATH))
                except OSError as e:
                    _load_error = f"cannot load {LIB_PATH}: {e}"
    if _lib is None:
        raise RuntimeError(_load_error)
    return _lib
