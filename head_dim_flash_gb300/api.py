"""PyTorch-facing API over the C ABI: tensors in, tensors out.

PyTorch only provides device memory, the current stream and autograd; every
step of the computation runs in the library's CUDA kernels. Nothing here
computes attention, and nothing falls back to another implementation: an
unsupported call raises (FFPA docs, "Backends Overview" page, "Automatic SDPA
fallback": unsupported dtype and similar raise NotImplementedError /
ValueError, no silent fallback).

Layouts (FFPA docs, "CuTe-DSL Backend" page): dense q [B, Hq, Nq, D],
k/v [B, Hkv, Nkv, D]; packed varlen q [Tq, Hq, D], k/v [Tk, Hkv, D] with
int32 cu_seqlens; LSE is fp32 [B, Hq, Nq] (dense) or [Hq, Tq] (varlen).

Dense tensors are passed as strided views (ffpa_view) with no copy whenever
the head dim is the innermost, unit-stride dimension and the other strides are
multiples of 8 elements: contiguous [B, H, N, D] tensors, ``x.transpose(1, 2)``
of a [B, N, H, D] projection output, slices of a fused QKV buffer. Any other
layout is copied to a contiguous tensor first. Dense outputs default to the
layout of the matching input (``torch.empty_like``). Varlen inputs are made
contiguous.
"""
from __future__ import annotations

import math

import torch

from . import _ffi

_DTYPES = {torch.bfloat16: _ffi.BF16, torch.float16: _ffi.FP16}


def _dt(x: torch.Tensor) -> int:
    if x.dtype not in _DTYPES:
        raise NotImplementedError(f"dtype {x.dtype}: only torch.bfloat16 and torch.float16 are supported")
    return _DTYPES[x.dtype]


def _prep(*xs):
    out = []
    for x in xs:
        if not x.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        out.append(x.contiguous())
    dt = out[0].dtype
    for x in out[1:]:
        if x.dtype != dt:
            raise ValueError(f"mixed dtypes {dt} and {x.dtype}")
    return out


def _viewable(x: torch.Tensor) -> bool:
    """True when the dense 4-D tensor can be handed to the kernels as an ffpa_view."""
    if x.dim() != 4 or x.stride(-1) != 1 or x.data_ptr() % 16 != 0:
        return False
    for size, stride in zip(x.shape[:3], x.stride()[:3]):
        if stride < 0 or stride % 8 != 0 or (size > 1 and stride == 0):
            return False
    return True


def _dense(*xs):
    """Dense inputs: checked, and copied only when no view of them fits the ABI."""
    out = []
    for x in xs:
        if not x.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        out.append(x if _viewable(x) else x.contiguous())
    dt = out[0].dtype
    for x in out[1:]:
        if x.dtype != dt:
            raise ValueError(f"mixed dtypes {dt} and {x.dtype}")
    return out


def _out_like(x: torch.Tensor) -> torch.Tensor:
    y = torch.empty_like(x)
    return y if _viewable(y) else torch.empty(x.shape, dtype=x.dtype, device=x.device)


def _view(x: torch.Tensor) -> _ffi.View:
    if not _viewable(x):
        raise ValueError(f"output of shape {tuple(x.shape)} and strides {x.stride()} is not an ffpa_view "
                         "(head dim innermost with unit stride, other strides multiples of 8 elements)")
    return _ffi.View(x.data_ptr(), x.stride(0), x.stride(1), x.stride(2))


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _scale(scale, D):
    return float(1.0 / math.sqrt(D)) if scale is None else float(scale)


# ----------------------------------------------------------------- dense
def fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None):
    """Dense forward through ffpa_fwd_strided (views, no copy). Returns (o, lse)."""
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,Hq,Nq,D], k and v [B,Hkv,Nkv,D]")
    q, k, v = _dense(q, k, v)
    B, Hq, Nq, D = q.shape
    Bk, Hkv, Nkv, Dk = k.shape
    if Bk != B or Dk != D:
        raise ValueError("q and k/v disagree on B or D")
    o = _out_like(q) if out is None else out
    l = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    if not l.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, Hq, Nq] tensor")
    st = _ffi.ffpa_fwd_strided(_dt(q), _view(q), _view(k), _view(v), _view(o), l.data_ptr(),
                               B, Hq, Hkv, Nq, Nkv, D, int(bool(causal)), _scale(scale, D), _stream())
    _ffi.raise_for(st, "ffpa_fwd_strided")
    return o, l


DECODE_ROWS = 16    # query rows of one kv head's group per decode CTA
DECODE_MAX_NQ = 8   # attention() sends Nq below this to the decode path


def decode_supported(q, k) -> bool:
    """True when ffpa_decode_fwd takes this problem (D % 64 == 0, grid within limits)."""
    B, Hq, Nq, D = q.shape
    Hkv = k.shape[1]
    if Hkv <= 0 or Hq % Hkv != 0 or D % 64 != 0:
        return False
    return B * Hkv * -(-(Hq // Hkv) * Nq // DECODE_ROWS) <= 65535 * 65535


def decode_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, workspace=None):
    """Decode / short-query forward through ffpa_decode_fwd (split over the keys).
    Same result as fwd(); raises NotImplementedError outside decode_supported()."""
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,Hq,Nq,D], k and v [B,Hkv,Nkv,D]")
    q, k, v = _dense(q, k, v)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    o = _out_like(q) if out is None else out
    l = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    ws_bytes = int(_ffi.ffpa_decode_workspace_bytes(_dt(q), B, Hq, Hkv, Nq, Nkv, D))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = _ffi.ffpa_decode_fwd(_dt(q), _view(q), _view(k), _view(v), _view(o), l.data_ptr(), workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), B, Hq, Hkv, Nq, Nkv, D,
                              int(bool(causal)), _scale(scale, D), _stream())
    _ffi.raise_for(st, "ffpa_decode_fwd")
    return o, l


def fp8_supported(D: int) -> bool:
    """Head dims of the FP8 forward: every multiple of 32 in [64, 1024]."""
    return D % 32 == 0 and 64 <= D <= 1024


def fp8_workspace(q, k):
    """Device scratch for fwd_fp8 (uint8, 256-byte aligned by the allocator)."""
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    n = int(_ffi.ffpa_fp8_workspace_bytes(B, Hq, Hkv, Nq, Nkv, D))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def _fp8_args(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,Hq,Nq,D], k and v [B,Hkv,Nkv,D]")
    return _dense(q, k, v)


def fp8_quantize(q, k, v, workspace=None):
    """Runs only the e4m3 quantization; returns (workspace, {name: view}) with
    q8, k8 (uint8 codes), v8t ([B, Hkv, D, ldv] codes of V^T) and the fp32 scales sq, sk, sv.
    The code views cover the D real columns; the workspace pads each code row
    to Dp = D rounded up to 128 with zero codes (q8_padded, k8_padded, v8t_padded)."""
    q, k, v = _fp8_args(q, k, v)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    ws = fp8_workspace(q, k) if workspace is None else workspace
    st = _ffi.ffpa_fp8_quantize(_dt(q), _view(q), _view(k), _view(v), ws.data_ptr(), ws.numel(),
                                B, Hq, Hkv, Nq, Nkv, D, _stream())
    _ffi.raise_for(st, "ffpa_fp8_quantize")
    off = _ffi.ffpa_fp8_workspace_layout(B, Hq, Hkv, Nq, Nkv, D)
    ldv = off[6]

    def region(i, n, shape, dtype=torch.uint8):
        t = ws[off[i]:off[i] + n * (4 if dtype == torch.float32 else 1)]
        return t.view(dtype).view(shape)

    Dp = (D + 127) // 128 * 128
    views = {
        "q8_padded": region(0, B * Hq * Nq * Dp, (B, Hq, Nq, Dp)),
        "k8_padded": region(1, B * Hkv * Nkv * Dp, (B, Hkv, Nkv, Dp)),
        "v8t_padded": region(2, B * Hkv * Dp * ldv, (B, Hkv, Dp, ldv)),
        "sq": region(3, B * Hq, (B, Hq), torch.float32),
        "sk": region(4, B * Hkv, (B, Hkv), torch.float32),
        "sv": region(5, B * Hkv, (B, Hkv), torch.float32),
    }
    views["q8"] = views["q8_padded"][..., :D]
    views["k8"] = views["k8_padded"][..., :D]
    views["v8t"] = views["v8t_padded"][:, :, :D]
    return ws, views


def fwd_fp8(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, workspace=None):
    """FP8 (e4m3) forward through ffpa_fwd_fp8: bf16/fp16 in, O in the input
    dtype and fp32 LSE out; D a multiple of 32 in [64, 1024]. Returns (o, lse)."""
    q, k, v = _fp8_args(q, k, v)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    o = _out_like(q) if out is None else out
    l = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    ws = fp8_workspace(q, k) if workspace is None else workspace
    st = _ffi.ffpa_fwd_fp8(_dt(q), _view(q), _view(k), _view(v), _view(o), l.data_ptr(), ws.data_ptr(), ws.numel(),
                           B, Hq, Hkv, Nq, Nkv, D, int(bool(causal)), _scale(scale, D), _stream())
    _ffi.raise_for(st, "ffpa_fwd_fp8")
    return o, l


def fwd_fp8_quantized(workspace, shape_q, shape_k, dtype, causal: bool = False, scale: float | None = None,
                      out=None, lse=None):
    """The FP8 attention alone, on a workspace that fp8_quantize filled for q of
    shape_q and k/v of shape_k (inputs quantized once, attended many times)."""
    B, Hq, Nq, D = shape_q
    _, Hkv, Nkv, _ = shape_k
    o = torch.empty(shape_q, dtype=dtype, device=workspace.device) if out is None else out
    l = torch.empty((B, Hq, Nq), dtype=torch.float32, device=workspace.device) if lse is None else lse
    st = _ffi.ffpa_fwd_fp8_quantized(_dt(o), _view(o), l.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                     B, Hq, Hkv, Nq, Nkv, D, int(bool(causal)), _scale(scale, D), _stream())
    _ffi.raise_for(st, "ffpa_fwd_fp8_quantized")
    return o, l


# Default cap of the backward workspace bwd() and varlen_bwd() allocate: the
# stored P^T / dS^T tiles of every head when they fit in it (8.6 GB at
# B1 H32 N8192 D512), else of as many kv groups per chunk as fit. A fixed
# size, so that the path a call takes never depends on what else is allocated.
BWD_WORKSPACE_BUDGET = 16 << 30


def bwd_workspace_bytes(q, k, causal: bool | None = None, budget: int | None = None) -> int:
    """Backward workspace bytes: the row statistics only (causal None); with
    room for the stored dS and P tiles of every head where that path applies
    (budget None: ffpa_bwd_workspace_bytes_ds); or the largest useful size
    within `budget` bytes (ffpa_bwd_workspace_bytes_budget: the tiles of every
    head, else of a chunk of kv groups, else the row statistics)."""
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    if causal is None:
        return int(_ffi.ffpa_bwd_workspace_bytes(_dt(q), B, Hq, Hkv, Nq, Nkv, D))
    if budget is None:
        return int(_ffi.ffpa_bwd_workspace_bytes_ds(_dt(q), B, Hq, Hkv, Nq, Nkv, D, int(bool(causal))))
    return int(_ffi.ffpa_bwd_workspace_bytes_budget(_dt(q), B, Hq, Hkv, Nq, Nkv, D, int(bool(causal)),
                                                     int(budget)))


def bwd_workspace(q, k, causal: bool, budget: int = BWD_WORKSPACE_BUDGET):
    """A backward workspace of the largest useful size within `budget` bytes."""
    n = bwd_workspace_bytes(q, k, causal, budget)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)


def bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, workspace=None,
        dq=None, dk=None, dv=None, stages: int = 15):
    """Dense backward through ffpa_bwd_strided (views, no copy), or ffpa_bwd_stages
    for a subset of its launches (bit 0 preprocess, bit 1 dV, bit 2 dQ, bit 3 dK,
    bit 4 dQ from the dS a dK stage stored, bit 5 dV storing P / dK reading it;
    contiguous tensors). Without a workspace, one of at most
    BWD_WORKSPACE_BUDGET bytes is allocated (bwd_workspace): the stored-tile
    path for every head, or in chunks of kv groups, where it applies. Returns
    (dq, dk, dv)."""
    q, k, v, o, dout = _dense(q, k, v, o, dout)
    lse = lse.contiguous()
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    if workspace is None:
        workspace = bwd_workspace(q, k, causal)
    dq = _out_like(q) if dq is None else dq
    dk = _out_like(k) if dk is None else dk
    dv = _out_like(v) if dv is None else dv
    tail = (workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            B, Hq, Hkv, Nq, Nkv, D, int(bool(causal)), _scale(scale, D))
    if stages == 15:
        st = _ffi.ffpa_bwd_strided(_dt(q), _view(q), _view(k), _view(v), _view(o), lse.data_ptr(), _view(dout),
                                   _view(dq), _view(dk), _view(dv), *tail, _stream())
        _ffi.raise_for(st, "ffpa_bwd_strided")
    else:
        ts = [x.contiguous() for x in (q, k, v, o, dout)]
        for name, x in (("dq", dq), ("dk", dk), ("dv", dv)):
            if not x.is_contiguous():
                raise ValueError(f"{name} must be contiguous when stages != 15")
        st = _ffi.ffpa_bwd_stages(_dt(q), *(x.data_ptr() for x in ts[:4]), lse.data_ptr(), ts[4].data_ptr(),
                                  dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), *tail, int(stages), _stream())
        _ffi.raise_for(st, "ffpa_bwd_stages")
    return dq, dk, dv


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale):
        # short queries (Nq < 8, decode) take the split-KV path; the backward
        # is the same either way (O and LSE have the same meaning)
        if q.dim() == 4 and 0 < q.shape[2] < DECODE_MAX_NQ and decode_supported(q, k):
            o, lse = decode_fwd(q, k, v, causal, scale)
        else:
            o, lse = fwd(q, k, v, causal, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale = causal, scale
        return o, lse

    @staticmethod
    def backward(ctx, do, dlse):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = bwd(q, k, v, o, lse, do, ctx.causal, ctx.scale)
        return dq, dk, dv, None, None


def attention(q, k, v, causal: bool = False, scale: float | None = None, return_lse: bool = False):
    """O = softmax(scale * Q K^T [bottom-right causal]) V, differentiable w.r.t. q, k, v.

    The gradient of the returned LSE is not propagated (it is an auxiliary output).
    """
    o, lse = _Attention.apply(q, k, v, bool(causal), scale)
    return (o, lse) if return_lse else o


# ----------------------------------------------------------------- varlen
def _cu(cu, device):
    if cu is None:
        return None
    if cu.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    return cu.to(device).contiguous()


def varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal=False, scale=None):
    """Packed forward through ffpa_varlen_fwd. Returns (o [Tq,Hq,D], lse [Hq,Tq])."""
    q, k, v = _prep(q, k, v)
    Tq, Hq, D = q.shape
    Tk, Hkv, _ = k.shape
    cq, ck = _cu(cu_seqlens_q, q.device), _cu(cu_seqlens_k, q.device)
    batch = cq.numel() - 1
    o = torch.empty_like(q)
    lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    st = _ffi.ffpa_varlen_fwd(_dt(q), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              cq.data_ptr(), ck.data_ptr(), batch, Tq, Tk, int(max_seqlen_q), int(max_seqlen_k),
                              Hq, Hkv, D, int(bool(causal)), _scale(scale, D), _stream())
    _ffi.raise_for(st, "ffpa_varlen_fwd")
    return o, lse


def varlen_fp8_workspace(q, k, cu_seqlens_q, max_seqlen_q, max_seqlen_k):
    """Device scratch for varlen_fwd_fp8 (uint8, 256-byte aligned by the allocator)."""
    Tq, Hq, D = q.shape
    Tk, Hkv, _ = k.shape
    batch = cu_seqlens_q.numel() - 1
    n = int(_ffi.ffpa_varlen_fp8_workspace_bytes(batch, Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def varlen_fwd_fp8(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal=False, scale=None,
                   workspace=None):
    """Packed FP8 (e4m3) forward through ffpa_varlen_fwd_fp8: each sequence quantized
    per head as fwd_fp8 quantizes a batch entry. Returns (o [Tq,Hq,D], lse [Hq,Tq])."""
    q, k, v = _prep(q, k, v)
    Tq, Hq, D = q.shape
    Tk, Hkv, _ = k.shape
    cq, ck = _cu(cu_seqlens_q, q.device), _cu(cu_seqlens_k, q.device)
    batch = cq.numel() - 1
    o = torch.empty_like(q)
    lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    ws = varlen_fp8_workspace(q, k, cq, max_seqlen_q, max_seqlen_k) if workspace is None else workspace
    st = _ffi.ffpa_varlen_fwd_fp8(_dt(q), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                  cq.data_ptr(), ck.data_ptr(), batch, Tq, Tk, int(max_seqlen_q), int(max_seqlen_k),
                                  Hq, Hkv, D, int(bool(causal)), _scale(scale, D), ws.data_ptr(), ws.numel(),
                                  _stream())
    _ffi.raise_for(st, "ffpa_varlen_fwd_fp8")
    return o, lse


def varlen_workspace_bytes(q, k, cu_seqlens_q, max_seqlen_q, max_seqlen_k, causal: bool,
                           budget: int = BWD_WORKSPACE_BUDGET) -> int:
    """Largest useful packed-backward workspace within `budget` bytes
    (ffpa_varlen_bwd_workspace_bytes_budget)."""
    Tq, Hq, D = q.shape
    Tk, Hkv, _ = k.shape
    batch = cu_seqlens_q.numel() - 1
    return int(_ffi.ffpa_varlen_bwd_workspace_bytes_budget(_dt(q), batch, Tq, Tk, int(max_seqlen_q),
                                                            int(max_seqlen_k), Hq, Hkv, D, int(bool(causal)),
                                                            int(budget)))


def varlen_bwd(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal=False,
               scale=None, workspace=None):
    """Packed backward through ffpa_varlen_bwd. Without a workspace, one of at
    most BWD_WORKSPACE_BUDGET bytes is allocated (the stored-tile path for
    every head, or in chunks of kv groups, where it applies). Returns
    (dq, dk, dv)."""
    q, k, v, o, dout = _prep(q, k, v, o, dout)
    lse = lse.contiguous()
    Tq, Hq, D = q.shape
    Tk, Hkv, _ = k.shape
    cq, ck = _cu(cu_seqlens_q, q.device), _cu(cu_seqlens_k, q.device)
    batch = cq.numel() - 1
    sizes = (_dt(q), batch, Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D)
    if workspace is None:
        n = int(_ffi.ffpa_varlen_bwd_workspace_bytes_budget(*sizes, int(bool(causal)), BWD_WORKSPACE_BUDGET))
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = _ffi.ffpa_varlen_bwd(_dt(q), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cq.data_ptr(),
                              ck.data_ptr(), batch, Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D,
                              int(bool(causal)), _scale(scale, D), workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), _stream())
    _ffi.raise_for(st, "ffpa_varlen_bwd")
    return dq, dk, dv


class _VarlenAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, cq, ck, mq, mk, causal, scale):
        o, lse = varlen_fwd(q, k, v, cq, ck, mq, mk, causal, scale)
        ctx.save_for_backward(q, k, v, o, lse, cq, ck)
        ctx.args = (mq, mk, causal, scale)
        return o, lse

    @staticmethod
    def backward(ctx, do, dlse):
        q, k, v, o, lse, cq, ck = ctx.saved_tensors
        mq, mk, causal, scale = ctx.args
        dq, dk, dv = varlen_bwd(q, k, v, o, lse, do, cq, ck, mq, mk, causal, scale)
        return dq, dk, dv, None, None, None, None, None, None


def varlen_attention(q, k, v, cu_seqlens_q, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None,
                     causal: bool = False, scale: float | None = None, return_lse: bool = False):
    """Packed-THD attention (FFPA docs, "CuTe-DSL Backend" page, "Varlen (packed THD) API").

    cu_seqlens_k=None means cu_seqlens_k = cu_seqlens_q. When max_seqlen_* is
    None it is read from cu_seqlens (one device-to-host copy).
    """
    if cu_seqlens_k is None:
        cu_seqlens_k = cu_seqlens_q
    if max_seqlen_q is None:
        max_seqlen_q = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if cu_seqlens_q.numel() > 1 else 0
    if max_seqlen_k is None:
        max_seqlen_k = int((cu_seqlens_k[1:] - cu_seqlens_k[:-1]).max().item()) if cu_seqlens_k.numel() > 1 else 0
    cq, ck = _cu(cu_seqlens_q, q.device), _cu(cu_seqlens_k, q.device)
    o, lse = _VarlenAttention.apply(q, k, v, cq, ck, int(max_seqlen_q), int(max_seqlen_k), bool(causal), scale)
    return (o, lse) if return_lse else o


def get_status() -> None:
    """Synchronises the current stream and raises if a kernel reported a device time-out."""
    _ffi.raise_for(_ffi.ffpa_get_status(_stream()), "device status")
