"""FP8 (e4m3) forward reference (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module. It shares no code with the CUDA library.

The FFPA docs ("Backends Overview" page, capability matrix and its notes)
list FP8 forward kernels that take fp16/bf16 Q/K/V and quantize them inside
the kernel; the pages give no scale granularity and no rounding rule. The
readings taken here (each one a plain choice the rest of the pages support):

* e4m3 is the OCP "fn" format: 4 exponent bits (bias 7), 3 mantissa bits,
  subnormals, no infinities, largest finite value 448. Conversion is
  round-to-nearest-even with saturation to +-448 (the hardware
  ``cvt.rn.satfinite`` rule).
* One scale per (batch, head) and tensor: amax = max |x| over the head's
  [N, D] slice (fp32), scale = amax / 448 and inv = 448 / amax, both rounded
  to fp32 (scale = inv = 1 for an all-zero head); code = e4m3(fp32(x * inv)).
* The attention is the plain definition (``attention_fwd``) applied to the
  dequantized inputs code * scale, in fp64. The kernel further rounds the
  softmax numerators P to e4m3 before the P V product (no extra scale);
  ``p_rounding_bound`` bounds what that rounding can change in O.
* A packed (THD) batch ("CuTe-DSL Backend", "Varlen (packed THD) API") is
  quantized and attended sequence by sequence, each sequence as one batch
  entry of the dense FP8 forward (``varlen_attention_fwd_fp8``); the pages'
  FP8 rows offer no packed layout, so this is the plain extension.
"""
from __future__ import annotations

import numpy as np

from . import attention_fwd

E4M3_MAX = 448.0
_MIN_NORMAL = 2.0 ** -6
_SUB_STEP = 2.0 ** -9


def e4m3_round(y) -> np.ndarray:
    """Values of fp32 inputs rounded to e4m3 (nearest, ties to even, saturating), as float64."""
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    a = np.abs(y)
    out = np.empty_like(a)
    normal = a >= _MIN_NORMAL
    # quantum of the binade: 2^(e - 3) for |y| in [2^e, 2^(e+1)); frexp gives |y| = m 2^x, m in [0.5, 1)
    _, ex = np.frexp(np.where(normal, a, 1.0))
    quantum = np.ldexp(1.0, ex - 1 - 3)
    out[normal] = np.rint(a[normal] / quantum[normal]) * quantum[normal]
    sub = ~normal
    out[sub] = np.rint(a[sub] / _SUB_STEP) * _SUB_STEP
    out = np.minimum(out, E4M3_MAX)
    return np.where(np.signbit(y), -out, out)


def e4m3_encode(values) -> np.ndarray:
    """uint8 codes of values that are exactly representable in e4m3 (sign kept for zeros)."""
    v = np.asarray(values, dtype=np.float64)
    a = np.abs(v)
    code = np.zeros(v.shape, dtype=np.int64)
    normal = a >= _MIN_NORMAL
    m, ex = np.frexp(np.where(normal, a, 1.0))
    e = ex - 1                                   # |v| = (1 + f) 2^e
    mant = np.rint((2.0 * m - 1.0) * 8.0).astype(np.int64)
    code = np.where(normal, ((e + 7) << 3) | mant, np.rint(a / _SUB_STEP).astype(np.int64))
    code = code | (np.signbit(v).astype(np.int64) << 7)
    return code.astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of uint8 e4m3 codes (0x7F / 0xFF, the NaN codes, decode to NaN)."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * _SUB_STEP, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def head_scales(x):
    """Per-(batch, head) (scale, inv) of a [B, H, N, D] tensor, as fp32 arrays [B, H]."""
    x32 = _f32(x)
    amax = np.abs(x32).max(axis=(2, 3)) if x32.size else np.zeros(x32.shape[:2], np.float32)
    amax = amax.astype(np.float32)
    pos = amax > 0
    scale = np.where(pos, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(pos, np.float32(E4M3_MAX) / np.where(pos, amax, np.float32(1.0)), np.float32(1.0))
    return scale, inv.astype(np.float32)


def quantize(x):
    """e4m3 codes [B, H, N, D] (uint8) and fp32 scales [B, H] of a bf16/fp16 tensor."""
    x32 = _f32(x)
    scale, inv = head_scales(x32)
    y = (x32 * inv[:, :, None, None]).astype(np.float32)  # one fp32 product, rounded to nearest
    return e4m3_encode(e4m3_round(y)), scale


def dequantize(codes, scale) -> np.ndarray:
    return e4m3_decode(codes) * np.asarray(scale, dtype=np.float64)[:, :, None, None]


def attention_fwd_fp8(q, k, v, causal: bool = False, scale: float | None = None):
    """(O, LSE) of the attention of the dequantized e4m3 inputs, fp64; plus the dequantized inputs."""
    qd = dequantize(*quantize(q))
    kd = dequantize(*quantize(k))
    vd = dequantize(*quantize(v))
    o, lse = attention_fwd(qd, kd, vd, causal, scale)
    return o, lse, (qd, kd, vd)


def varlen_attention_fwd_fp8(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool = False, scale: float | None = None):
    """Packed FP8 forward: q [Tq, Hq, D], k/v [Tk, Hkv, D], int cu_seqlens [batch + 1].
    Each sequence is one batch entry of ``attention_fwd_fp8`` (its own per-head
    scales). Returns (O [Tq, Hq, D], LSE [Hq, Tq], bound [Tq, Hq, D]) with the
    ``p_rounding_bound`` of each sequence in ``bound``."""
    q32, k32, v32 = _f32(q), _f32(k), _f32(v)
    cq = np.asarray(cu_seqlens_q, dtype=np.int64)
    ck = np.asarray(cu_seqlens_k, dtype=np.int64)
    Tq, Hq, D = q32.shape
    o = np.zeros((Tq, Hq, D))
    lse = np.full((Hq, Tq), -np.inf)
    bound = np.zeros((Tq, Hq, D))
    sc = 1.0 / np.sqrt(D) if scale is None else float(scale)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        if q1 == q0:
            continue
        qb = q32[q0:q1].transpose(1, 0, 2)[None]  # [1, Hq, Lq, D]
        kb = k32[k0:k1].transpose(1, 0, 2)[None]
        vb = v32[k0:k1].transpose(1, 0, 2)[None]
        ob, lb, (qd, kd, vd) = attention_fwd_fp8(qb, kb, vb, causal, sc)
        o[q0:q1] = ob[0].transpose(1, 0, 2)
        lse[:, q0:q1] = lb[0]
        if k1 > k0:  # no keys: no P to round (O = 0 exactly)
            bound[q0:q1] = p_rounding_bound(qd, kd, vd, causal, sc)[0].transpose(1, 0, 2)
    return o, lse, bound


def p_rounding_bound(qd, kd, vd, causal: bool = False, scale: float | None = None) -> np.ndarray:
    """Element-wise bound on |O' - O| when each softmax numerator P_ij (taken
    relative to any reference m with row max - 8 <= m <= row max, in log2
    units, as a lazily rescaled online softmax keeps it) is rounded to e4m3
    before the P V product, O' = sum_j e4m3(P_ij) v_j / sum_j P_ij:

        |e4m3(P) - P| <= 2^-4 P + 2^-10  (half a unit in the last place:
        relative 2^-4 for normal values, absolute 2^-10 below 2^-6), so

        |O'_id - O_id| <= 2^-4 sum_j w_ij |v_jd| + 2^-10 sum_j |v_jd| / L_i,

    w = softmax weights, L_i = sum_j exp(s_ij - max_j s_ij) >= 1 over the
    legal keys (the 2^-10 term is largest, and taken, for m = row max).
    """
    qd, kd, vd = (np.asarray(t, dtype=np.float64) for t in (qd, kd, vd))
    B, Hq, Nq, D = qd.shape
    Hkv, Nkv = kd.shape[1], kd.shape[2]
    G = Hq // Hkv
    sc = 1.0 / np.sqrt(D) if scale is None else float(scale)
    wabs, _ = attention_fwd(qd, kd, np.abs(vd), causal, sc)
    bound = np.zeros((B, Hq, Nq, D))
    off = Nkv - Nq
    legal = np.ones((Nq, Nkv), dtype=bool)
    if causal:
        legal = np.arange(Nkv)[None, :] <= np.arange(Nq)[:, None] + off
    for b in range(B):
        for h in range(Hq):
            s = sc * qd[b, h] @ kd[b, h // G].T
            s = np.where(legal, s, -np.inf)
            mx = s.max(axis=1, keepdims=True)
            has = np.isfinite(mx[:, 0])
            ok = legal & has[:, None]
            el = np.where(ok, np.exp(np.where(ok, s - np.where(has[:, None], mx, 0.0), -np.inf)), 0.0)
            L = el.sum(axis=1)
            vsum = legal.astype(np.float64) @ np.abs(vd[b, h // G])   # sum over legal keys of |v|
            with np.errstate(divide="ignore", invalid="ignore"):
                term = np.where(has[:, None], vsum / np.where(L > 0, L, 1.0)[:, None], 0.0)
            bound[b, h] = 2.0 ** -4 * wabs[b, h] + 2.0 ** -10 * term
    return bound


def _f32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float32)
