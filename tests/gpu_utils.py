"""Helpers for the GPU parity tests: guarded output buffers and comparisons.

Tolerances (for bf16/fp16 inputs): O max-abs <= 2e-2; LSE max-abs <= 1e-3
with -inf matching exactly; dQ/dK/dV max-abs <= 5e-2 * max|grad| per tensor.
The relative Frobenius error is reported alongside (not gated) because a
nearly flat softmax makes |O| small.
"""
from __future__ import annotations

import numpy as np
import torch

O_TOL = 2e-2
LSE_TOL = 1e-3
GRAD_REL_TOL = 5e-2
GUARD = 4096  # elements of canary on each side of every output
ZERO_REF_ABS_TOL = 1e-4


class Guarded:
    """An output tensor carved from a larger buffer whose margins hold a
    sentinel; the body is pre-filled with NaN so unwritten elements show."""

    def __init__(self, shape, dtype, device="cuda"):
        n = int(np.prod(shape)) if len(shape) else 1
        self.buf = torch.empty(n + 2 * GUARD, dtype=dtype, device=device)
        self.sentinel = -12345.0 if dtype != torch.uint8 else 77
        self.buf[:GUARD].fill_(self.sentinel)
        self.buf[GUARD + n:].fill_(self.sentinel)
        self.n = n
        self.ref_lo = self.buf[:GUARD].clone()
        self.ref_hi = self.buf[GUARD + n:].clone()
        self.t = self.buf[GUARD:GUARD + n].view(shape)
        if dtype.is_floating_point:
            self.t.fill_(float("nan"))

    def check_guards(self, name):
        lo = self.buf[:GUARD]
        hi = self.buf[GUARD + self.n:]
        assert torch.equal(lo, self.ref_lo) and torch.equal(hi, self.ref_hi), f"{name}: write outside bounds"


def to64(x):
    return x.detach().float().cpu().double().numpy() if isinstance(x, torch.Tensor) else np.asarray(x, np.float64)


def check_o(o_gpu, o_ref, what="O"):
    o = to64(o_gpu)
    assert np.all(np.isfinite(o)), f"{what}: non-finite values"
    err = float(np.abs(o - o_ref).max()) if o.size else 0.0
    rel = float(np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-30)) if o.size else 0.0
    assert err <= O_TOL, f"{what} max-abs {err:.3e} > {O_TOL} (rel frob {rel:.2e})"
    return err, rel


def check_lse(lse_gpu, lse_ref, what="LSE"):
    l = to64(lse_gpu)
    ninf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(l), ninf_ref), f"{what}: -inf pattern differs"
    fin = ~ninf_ref
    assert np.all(np.isfinite(l[fin])), f"{what}: non-finite values"
    err = float(np.abs(l[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    assert err <= LSE_TOL, f"{what} max-abs {err:.3e} > {LSE_TOL}"
    return err


def check_grad(g_gpu, g_ref, what):
    g = to64(g_gpu)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    scale = float(np.abs(g_ref).max()) if g_ref.size else 0.0
    err = float(np.abs(g - g_ref).max()) if g.size else 0.0
    bound = GRAD_REL_TOL * scale
    rel = float(np.linalg.norm(g - g_ref) / max(np.linalg.norm(g_ref), 1e-30)) if g.size else 0.0
    if scale == 0.0:
        # an all-zero reference that is zero by cancellation (e.g. one legal
        # key: dS = P (dP - delta) = 0) is reached only up to rounding
        bound = ZERO_REF_ABS_TOL
    assert err <= bound, f"{what} max-abs {err:.3e} > {bound:.3e} (rel frob {rel:.2e})"
    return err, rel


def check_empty_rows_exact(o, lse, dq, empty_mask):
    """Rows without a legal key: O = 0, LSE = -inf and dQ = 0 exactly."""
    o, lse, dq = to64(o), to64(lse), to64(dq) if dq is not None else None
    assert np.all(o[empty_mask] == 0.0), "O not exactly zero on rows without a legal key"
    assert np.all(np.isneginf(lse[empty_mask])), "LSE not -inf on rows without a legal key"
    if dq is not None:
        assert np.all(dq[empty_mask] == 0.0), "dQ not exactly zero on rows without a legal key"
