"""ctypes binding of the C ABI in ``include/ffpa.h`` (argument marshalling only).

Every function here has the C name and argument order. The shared library is
built in-tree by ``head_dim_flash_gb300.build`` into ``_lib/libffpa.so``; if it
is missing, loading raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libffpa.so")

OK, ERR_INVALID_VALUE, ERR_NOT_SUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
BF16, FP16 = 0, 1

# Every symbol the header declares (checked by the ABI tests).
EXPORTS = (
    "ffpa_fwd",
    "ffpa_fwd_strided",
    "ffpa_bwd_workspace_bytes",
    "ffpa_bwd",
    "ffpa_bwd_strided",
    "ffpa_decode_workspace_bytes",
    "ffpa_decode_fwd",
    "ffpa_bwd_workspace_bytes_ds",
    "ffpa_bwd_workspace_bytes_budget",
    "ffpa_fp8_workspace_bytes",
    "ffpa_fp8_workspace_layout",
    "ffpa_fp8_quantize",
    "ffpa_fwd_fp8",
    "ffpa_fwd_fp8_quantized",
    "ffpa_varlen_fp8_workspace_bytes",
    "ffpa_varlen_fwd_fp8",
    "ffpa_bwd_stages",
    "ffpa_bwd_noalloc",
    "ffpa_varlen_fwd",
    "ffpa_varlen_bwd_workspace_bytes",
    "ffpa_varlen_bwd_workspace_bytes_ds",
    "ffpa_varlen_bwd_workspace_bytes_budget",
    "ffpa_varlen_bwd",
    "ffpa_get_status",
    "ffpa_last_error",
    "ffpa_set_wait_limit_ns",
    "ffpa_selftest_wait_timeout",
    "ffpa_num_sms",
)

_lock = threading.Lock()
_lib = None

_i = ctypes.c_int
_f = ctypes.c_float
_p = ctypes.c_void_p
_sz = ctypes.c_size_t
_u64 = ctypes.c_uint64


class View(ctypes.Structure):
    """``ffpa_view``: data pointer and element strides of a [B, H, N, D] tensor."""

    _fields_ = [("data", ctypes.c_void_p), ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64),
                ("stride_n", ctypes.c_int64)]


def _declare(lib):
    lib.ffpa_fwd.argtypes = [_i, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p]
    lib.ffpa_fwd.restype = _i
    lib.ffpa_fwd_strided.argtypes = [_i, View, View, View, View, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p]
    lib.ffpa_fwd_strided.restype = _i
    lib.ffpa_bwd_strided.argtypes = [_i, View, View, View, View, _p, View, View, View, View, _p, _sz, _i, _i, _i, _i,
                                     _i, _i, _i, _f, _p]
    lib.ffpa_bwd_strided.restype = _i
    lib.ffpa_bwd_workspace_bytes_ds.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i]
    lib.ffpa_bwd_workspace_bytes_ds.restype = _sz
    lib.ffpa_bwd_workspace_bytes_budget.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _sz]
    lib.ffpa_bwd_workspace_bytes_budget.restype = _sz
    lib.ffpa_fp8_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i]
    lib.ffpa_fp8_workspace_bytes.restype = _sz
    lib.ffpa_fp8_workspace_layout.argtypes = [_i, _i, _i, _i, _i, _i, ctypes.POINTER(_sz)]
    lib.ffpa_fp8_workspace_layout.restype = _sz
    lib.ffpa_fp8_quantize.argtypes = [_i, View, View, View, _p, _sz, _i, _i, _i, _i, _i, _i, _p]
    lib.ffpa_fp8_quantize.restype = _i
    lib.ffpa_fwd_fp8.argtypes = [_i, View, View, View, View, _p, _p, _sz, _i, _i, _i, _i, _i, _i, _i, _f, _p]
    lib.ffpa_fwd_fp8.restype = _i
    lib.ffpa_fwd_fp8_quantized.argtypes = [_i, View, _p, _p, _sz, _i, _i, _i, _i, _i, _i, _i, _f, _p]
    lib.ffpa_fwd_fp8_quantized.restype = _i
    lib.ffpa_varlen_fp8_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i]
    lib.ffpa_varlen_fp8_workspace_bytes.restype = _sz
    lib.ffpa_varlen_fwd_fp8.argtypes = [_i, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f, _p,
                                        _sz, _p]
    lib.ffpa_varlen_fwd_fp8.restype = _i
    lib.ffpa_decode_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i]
    lib.ffpa_decode_workspace_bytes.restype = _sz
    lib.ffpa_decode_fwd.argtypes = [_i, View, View, View, View, _p, _p, _sz, _i, _i, _i, _i, _i, _i, _i, _f, _p]
    lib.ffpa_decode_fwd.restype = _i
    lib.ffpa_bwd_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i]
    lib.ffpa_bwd_workspace_bytes.restype = _sz
    lib.ffpa_bwd.argtypes = [_i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _sz, _i, _i, _i, _i, _i, _i, _i, _f, _p]
    lib.ffpa_bwd.restype = _i
    lib.ffpa_bwd_stages.argtypes = [_i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _sz, _i, _i, _i, _i, _i, _i, _i, _f,
                                    ctypes.c_uint, _p]
    lib.ffpa_bwd_stages.restype = _i
    lib.ffpa_bwd_noalloc.argtypes = [_i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p]
    lib.ffpa_bwd_noalloc.restype = _i
    lib.ffpa_varlen_fwd.argtypes = [_i, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f, _p]
    lib.ffpa_varlen_fwd.restype = _i
    lib.ffpa_varlen_bwd_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _i]
    lib.ffpa_varlen_bwd_workspace_bytes.restype = _sz
    lib.ffpa_varlen_bwd_workspace_bytes_ds.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _i, _i]
    lib.ffpa_varlen_bwd_workspace_bytes_ds.restype = _sz
    lib.ffpa_varlen_bwd_workspace_bytes_budget.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _sz]
    lib.ffpa_varlen_bwd_workspace_bytes_budget.restype = _sz
    lib.ffpa_varlen_bwd.argtypes = [_i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i,
                                    _i, _f, _p, _sz, _p]
    lib.ffpa_varlen_bwd.restype = _i
    lib.ffpa_get_status.argtypes = [_p]
    lib.ffpa_get_status.restype = _i
    lib.ffpa_last_error.argtypes = []
    lib.ffpa_last_error.restype = ctypes.c_char_p
    lib.ffpa_set_wait_limit_ns.argtypes = [_u64]
    lib.ffpa_set_wait_limit_ns.restype = None
    lib.ffpa_selftest_wait_timeout.argtypes = [_u64, _p]
    lib.ffpa_selftest_wait_timeout.restype = _i
    lib.ffpa_num_sms.argtypes = []
    lib.ffpa_num_sms.restype = _i
    return lib


def load(path: str | None = None):
    """Loads (once) and returns the CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"CUDA library {p} is missing: build it with "
                    "`python -m head_dim_flash_gb300.build` (nvcc, sm_103a)")
            lib = _declare(ctypes.CDLL(p))
            if path is not None:
                return lib
            _lib = lib
    return _lib


def last_error() -> str:
    return load().ffpa_last_error().decode(errors="replace")


def raise_for(status: int, what: str) -> None:
    """Maps a status code to the Python exception the API contract names."""
    if status == OK:
        return
    msg = f"{what}: {last_error()}"
    if status == ERR_NOT_SUPPORTED:
        raise NotImplementedError(msg)
    if status == ERR_INVALID_VALUE:
        raise ValueError(msg)
    if status == ERR_TIMEOUT:
        raise TimeoutError(msg)
    raise RuntimeError(msg)


# Thin wrappers with the C names (pointers are ints).
def ffpa_fwd(*args):
    return load().ffpa_fwd(*args)


def ffpa_fwd_strided(*args):
    return load().ffpa_fwd_strided(*args)


def ffpa_bwd_strided(*args):
    return load().ffpa_bwd_strided(*args)


def ffpa_bwd_workspace_bytes_ds(*args):
    return load().ffpa_bwd_workspace_bytes_ds(*args)


def ffpa_bwd_workspace_bytes_budget(*args):
    return load().ffpa_bwd_workspace_bytes_budget(*args)


def ffpa_fp8_workspace_bytes(*args):
    return load().ffpa_fp8_workspace_bytes(*args)


def ffpa_fp8_workspace_layout(B, Hq, Hkv, Nq, Nkv, D):
    """Byte offsets (q8, k8, v8t, sq, sk, sv), ldv and the total size of the FP8 workspace."""
    off = (_sz * 8)()
    load().ffpa_fp8_workspace_layout(B, Hq, Hkv, Nq, Nkv, D, off)
    return list(off)


def ffpa_fp8_quantize(*args):
    return load().ffpa_fp8_quantize(*args)


def ffpa_fwd_fp8(*args):
    return load().ffpa_fwd_fp8(*args)


def ffpa_fwd_fp8_quantized(*args):
    return load().ffpa_fwd_fp8_quantized(*args)


def ffpa_varlen_fp8_workspace_bytes(*args):
    return load().ffpa_varlen_fp8_workspace_bytes(*args)


def ffpa_varlen_fwd_fp8(*args):
    return load().ffpa_varlen_fwd_fp8(*args)


def ffpa_decode_workspace_bytes(*args):
    return load().ffpa_decode_workspace_bytes(*args)


def ffpa_decode_fwd(*args):
    return load().ffpa_decode_fwd(*args)


def ffpa_bwd_workspace_bytes(*args):
    return load().ffpa_bwd_workspace_bytes(*args)


def ffpa_bwd(*args):
    return load().ffpa_bwd(*args)


def ffpa_bwd_stages(*args):
    return load().ffpa_bwd_stages(*args)


def ffpa_bwd_noalloc(*args):
    return load().ffpa_bwd_noalloc(*args)


def ffpa_varlen_fwd(*args):
    return load().ffpa_varlen_fwd(*args)


def ffpa_varlen_bwd_workspace_bytes(*args):
    return load().ffpa_varlen_bwd_workspace_bytes(*args)


def ffpa_varlen_bwd_workspace_bytes_ds(*args):
    return load().ffpa_varlen_bwd_workspace_bytes_ds(*args)


def ffpa_varlen_bwd_workspace_bytes_budget(*args):
    return load().ffpa_varlen_bwd_workspace_bytes_budget(*args)


def ffpa_varlen_bwd(*args):
    return load().ffpa_varlen_bwd(*args)


def ffpa_get_status(stream):
    return load().ffpa_get_status(stream)


def ffpa_last_error():
    return load().ffpa_last_error()


def ffpa_set_wait_limit_ns(ns):
    return load().ffpa_set_wait_limit_ns(ns)


def ffpa_selftest_wait_timeout(limit_ns, stream):
    return load().ffpa_selftest_wait_timeout(limit_ns, stream)


def ffpa_num_sms():
    return load().ffpa_num_sms()
