"""fp64 CPU oracle for exact softmax attention (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it, and it
shares no code with the CUDA library.

The arithmetic lives in ``attention_oracle.c`` (plain two-pass softmax per
query row in fp64, following the FFPA docs, "CuTe-DSL Backend" page, sections
"Hard constraints" and "Varlen (packed THD) API"). This module compiles it
with gcc on first use and marshals numpy arrays through ctypes.

Every function takes the inputs exactly as the GPU sees them (bf16/fp16
tensors or any array) and widens them to fp64 first.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)
_lp = ctypes.POINTER(ctypes.c_long)
_L = ctypes.c_long


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle (default: ``oracle/_build/liboracle.so``) with portable flags."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    stale = (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src)
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", "-Wall", "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def load_library(path: str):
    """Loads a compiled oracle and declares its C signatures."""
    lib = ctypes.CDLL(path)
    lib.ffpa_oracle_fwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _L, _L, _L, _L, _L, _L, ctypes.c_int, ctypes.c_double]
    lib.ffpa_oracle_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _L, _L, _L, _L, _L, _L, ctypes.c_int, ctypes.c_double]
    lib.ffpa_oracle_varlen_fwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _ip, _ip, _L, _L, _L, _L, _L, ctypes.c_int, ctypes.c_double]
    lib.ffpa_oracle_varlen_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _ip, _ip, _L, _L, _L, _L, _L, ctypes.c_int, ctypes.c_double]
    lib.ffpa_oracle_fwd_rows.argtypes = [_dp, _dp, _dp, _lp, _L, _dp, _dp, _L, _L, _L, ctypes.c_int, ctypes.c_double]
    lib.ffpa_oracle_num_threads.restype = ctypes.c_int
    lib.ffpa_oracle_set_num_threads.argtypes = [ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def use_library(lib) -> None:
    """Points this module at another compiled oracle (``None`` restores the default)."""
    global _lib
    with _lock:
        _lib = lib


def _f64(x) -> np.ndarray:
    """Exact widening of any tensor/array to a contiguous fp64 numpy array."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.int32).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def num_threads() -> int:
    return int(_load().ffpa_oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().ffpa_oracle_set_num_threads(int(n))


def _check_group(hq: int, hkv: int) -> None:
    if hkv <= 0 or hq % hkv:
        raise ValueError(f"Hq={hq} must be a positive multiple of Hkv={hkv}")


def attention_fwd(q, k, v, causal: bool = False, scale: float | None = None):
    """Dense forward. q [B,Hq,Nq,D], k/v [B,Hkv,Nkv,D] -> (O [B,Hq,Nq,D], LSE [B,Hq,Nq]) in fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    _check_group(Hq, Hkv)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, Nq), dtype=np.float64)
    _load().ffpa_oracle_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), B, Hq, Hkv, Nq, Nkv, D, int(bool(causal)), float(scale))
    return o, lse


def attention_bwd(q, k, v, dout, causal: bool = False, scale: float | None = None):
    """Dense backward of L = sum(dO*O). Returns (dQ, dK, dV) in fp64."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    _check_group(Hq, Hkv)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    _load().ffpa_oracle_bwd(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv),
                            B, Hq, Hkv, Nq, Nkv, D, int(bool(causal)), float(scale))
    return dq, dk, dv


def varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k=None, causal: bool = False, scale: float | None = None):
    """Packed THD forward. q [Tq,Hq,D], k/v [Tk,Hkv,D] -> (O [Tq,Hq,D], LSE [Hq,Tq])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu_q = _i32(cu_seqlens_q)
    cu_k = cu_q if cu_seqlens_k is None else _i32(cu_seqlens_k)
    Tq, Hq, D = q.shape
    _, Hkv, _ = k.shape
    _check_group(Hq, Hkv)
    batch = cu_q.shape[0] - 1
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.zeros_like(q)
    lse = np.zeros((Hq, Tq), dtype=np.float64)
    _load().ffpa_oracle_varlen_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), cu_q.ctypes.data_as(_ip), cu_k.ctypes.data_as(_ip),
                                   batch, Tq, Hq, Hkv, D, int(bool(causal)), float(scale))
    return o, lse


def varlen_bwd(q, k, v, dout, cu_seqlens_q, cu_seqlens_k=None, causal: bool = False, scale: float | None = None):
    """Packed THD backward. Returns (dQ [Tq,Hq,D], dK [Tk,Hkv,D], dV [Tk,Hkv,D])."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    cu_q = _i32(cu_seqlens_q)
    cu_k = cu_q if cu_seqlens_k is None else _i32(cu_seqlens_k)
    Tq, Hq, D = q.shape
    _, Hkv, _ = k.shape
    _check_group(Hq, Hkv)
    batch = cu_q.shape[0] - 1
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    _load().ffpa_oracle_varlen_bwd(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv),
                                   cu_q.ctypes.data_as(_ip), cu_k.ctypes.data_as(_ip),
                                   batch, Tq, Hq, Hkv, D, int(bool(causal)), float(scale))
    return dq, dk, dv


def attention_fwd_rows(q_head, k_head, v_head, rows, causal: bool = False, scale: float | None = None):
    """Forward of selected query rows of ONE dense head.

    q_head [Nq,D], k_head/v_head [Nkv,D], rows: iterable of row indices.
    Returns (O [n,D], LSE [n]). Used to check or time a bounded sample.
    """
    q, k, v = _f64(q_head), _f64(k_head), _f64(v_head)
    Nq, D = q.shape
    Nkv = k.shape[0]
    r = np.ascontiguousarray(np.asarray(list(rows), dtype=np.int64))
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.zeros((r.shape[0], D), dtype=np.float64)
    lse = np.zeros((r.shape[0],), dtype=np.float64)
    _load().ffpa_oracle_fwd_rows(_p(q), _p(k), _p(v), r.ctypes.data_as(_lp), r.shape[0], _p(o), _p(lse),
                                 Nq, Nkv, D, int(bool(causal)), float(scale))
    return o, lse
