"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic. Tests, the smoke check and ``bench.py`` use it to feed
the CUDA library and the oracle the same bytes.

Recipe: a CPU ``torch.Generator`` seeded per workload draws fp32 standard
normals in the order q, k, v, dO; each is multiplied by the workload's
amplitude and rounded (round-to-nearest-even) to the workload's dtype.
Dense tensors are contiguous [B, H, N, D]; packed varlen tensors are
[T, H, D] with int32 cu_seqlens.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nkv: int
    D: int
    dtype: torch.dtype
    causal: bool
    seed: int
    amplitude: float = 1.0
    # varlen: per-sequence lengths (cu_seqlens_k = cu_seqlens_q); empty for dense
    seqlens: tuple = field(default_factory=tuple)

    @property
    def varlen(self) -> bool:
        return len(self.seqlens) > 0

    @property
    def scale(self) -> float:
        return 1.0 / (self.D ** 0.5)


def varlen_lengths(seed: int = 4, n: int = 6, lo: int = 512, hi: int = 6144) -> tuple:
    """Sequence lengths drawn uniformly in [lo, hi] from their own generator."""
    g = torch.Generator().manual_seed(seed)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g))


def cu_seqlens(lengths) -> torch.Tensor:
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return torch.tensor(out, dtype=torch.int32)


# The five workloads: a tiny single-head case, the D=512 N=8192 headline, a
# causal GQA cross-attention case, a head-dim sweep at non-tile-aligned N, and
# a packed varlen batch.
TINY = Workload("tiny B1 H1 N512 D512 bf16", 1, 1, 1, 512, 512, 512, torch.bfloat16, False, 0)
HEADLINE = Workload("dense B1 H32 N8192 D512 bf16", 1, 32, 32, 8192, 8192, 512, torch.bfloat16, False, 1)
GQA_CAUSAL = Workload("causal GQA B2 Hq32 Hkv8 Nq4096 Nkv8192 D512 bf16", 2, 32, 8, 4096, 8192, 512,
                      torch.bfloat16, True, 2)


def sweep(D: int) -> Workload:
    return Workload(f"sweep B1 H16 N4000 D{D} fp16", 1, 16, 16, 4000, 4000, D, torch.float16, False, 3, 0.5)


SWEEP = tuple(sweep(d) for d in (320, 640, 1024))
_VL = varlen_lengths()
VARLEN = Workload("varlen 6 seqs H32 D512 bf16 causal", len(_VL), 32, 32, max(_VL), max(_VL), 512,
                  torch.bfloat16, True, 40, 1.0, _VL)

ALL = (TINY, HEADLINE, GQA_CAUSAL) + SWEEP + (VARLEN,)

# Decode / short-query forward: one new query row per sequence against a long
# key cache, eight query heads per kv head (the split-KV path).
DECODE = Workload("decode B8 Hq32 Hkv8 Nq1 Nkv16384 D512 bf16", 8, 32, 8, 1, 16384, 512, torch.bfloat16, False, 50)

# FP8 forward: the dense headline shape and inputs, quantized to e4m3 for the kernel.
FP8 = Workload("fp8 forward dense B1 H32 N8192 D512 (bf16 in, e4m3 compute)", 1, 32, 32, 8192, 8192, 512,
               torch.bfloat16, False, 1)


def make_inputs(w: Workload, with_grad_out: bool = True):
    """Returns dict with q, k, v (and dO) as CPU tensors of w.dtype (+ cu_seqlens for varlen)."""
    g = torch.Generator().manual_seed(w.seed)
    if w.varlen:
        T = sum(w.seqlens)
        qs, ks = (T, w.Hq, w.D), (T, w.Hkv, w.D)
    else:
        qs, ks = (w.B, w.Hq, w.Nq, w.D), (w.B, w.Hkv, w.Nkv, w.D)
    out = {}
    for name, shape in (("q", qs), ("k", ks), ("v", ks)) + ((("dO", qs),) if with_grad_out else ()):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if w.amplitude != 1.0:
            x.mul_(w.amplitude)
        out[name] = x.to(w.dtype)
    if w.varlen:
        out["cu_seqlens"] = cu_seqlens(w.seqlens)
    return out


def random_dense(B, Hq, Hkv, Nq, Nkv, D, dtype=torch.bfloat16, seed=0, amplitude=1.0, with_grad_out=True):
    """Ad-hoc dense inputs (same recipe) for edge-case tests."""
    w = Workload("adhoc", B, Hq, Hkv, Nq, Nkv, D, dtype, False, seed, amplitude)
    return make_inputs(w, with_grad_out)


def random_varlen(lengths_q, lengths_k, Hq, Hkv, D, dtype=torch.bfloat16, seed=0, amplitude=1.0):
    """Ad-hoc packed inputs with separate q/k lengths (cu_seqlens_q, cu_seqlens_k)."""
    g = torch.Generator().manual_seed(seed)
    Tq, Tk = sum(lengths_q), sum(lengths_k)
    out = {}
    for name, shape in (("q", (Tq, Hq, D)), ("k", (Tk, Hkv, D)), ("v", (Tk, Hkv, D)), ("dO", (Tq, Hq, D))):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if amplitude != 1.0:
            x.mul_(amplitude)
        out[name] = x.to(dtype)
    out["cu_seqlens_q"] = cu_seqlens(lengths_q)
    out["cu_seqlens_k"] = cu_seqlens(lengths_k)
    return out
