"""GPU parity of the strided (zero-copy) dense calls against the fp64 oracle.

Inputs live in [B, N, H, D] storage or in a fused QKV buffer and reach the
kernels as ffpa_view strides; outputs are written into views of larger
buffers whose other entries must stay untouched. Both kernel families (CTA
pairs, one CTA per slab) run on both head dims.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from head_dim_flash_gb300 import api
from head_dim_flash_gb300 import workloads
from tests.gpu_utils import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_dim_flash_gb300 import build

    build.build()
    oracle.build()


def bnhd(x):
    """[B, H, N, D] values stored as [B, N, H, D] on the GPU, returned as the [B, H, N, D] view."""
    return x.transpose(1, 2).contiguous().cuda().transpose(1, 2)


@pytest.mark.parametrize("family", ["single", "pair"])
@pytest.mark.parametrize("D,causal", [(512, True), (320, False)])
def test_bnhd_views(family, D, causal, monkeypatch):
    monkeypatch.setenv("FFPA_KERNEL", family)
    B, Hq, Hkv, Nq, Nkv = 2, 4, 2, 150, 333
    inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, torch.float16, seed=60 + D, amplitude=0.5)
    q, k, v, do = (bnhd(inp[n]) for n in ("q", "k", "v", "dO"))
    scale = 1 / math.sqrt(D)
    o, lse = api.fwd(q, k, v, causal, scale)
    assert o.stride() == q.stride()  # the output keeps the [B, N, H, D] storage
    api.get_status()
    o_ref, lse_ref = oracle.attention_fwd(inp["q"], inp["k"], inp["v"], causal, scale)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    dq, dk, dv = api.bwd(q, k, v, o, lse, do, causal, scale)
    assert dq.stride() == q.stride() and dk.stride() == k.stride()
    api.get_status()
    g_ref = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], causal, scale)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv), g_ref):
        check_grad(got, ref, name)


@pytest.mark.parametrize("family", ["single", "pair"])
def test_fused_qkv_and_strided_outputs(family, monkeypatch):
    monkeypatch.setenv("FFPA_KERNEL", family)
    B, H, N, D = 1, 3, 200, 512
    inp = workloads.random_dense(B, H, H, N, N, D, torch.bfloat16, seed=70)
    fused = torch.empty(B, N, 3, H, D, dtype=torch.bfloat16, device="cuda")
    for i, n in enumerate(("q", "k", "v")):
        fused[:, :, i] = inp[n].transpose(1, 2).cuda()
    q, k, v = (fused[:, :, i].transpose(1, 2) for i in range(3))
    do = bnhd(inp["dO"])
    scale = 1 / math.sqrt(D)
    # outputs: slot 0 of [B, N, 2, H, D] buffers pre-filled with NaN; slot 1 must stay NaN
    bufs = {n: torch.full((B, N, 2, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
            for n in ("o", "dq", "dk", "dv")}
    views = {n: b[:, :, 0].transpose(1, 2) for n, b in bufs.items()}
    o, lse = api.fwd(q, k, v, True, scale, out=views["o"])
    dq, dk, dv = api.bwd(q, k, v, o, lse, do, True, scale, dq=views["dq"], dk=views["dk"], dv=views["dv"])
    api.get_status()
    for n, b in bufs.items():
        assert torch.isnan(b[:, :, 1].float()).all(), f"{n}: a store left its view"
    o_ref, lse_ref = oracle.attention_fwd(inp["q"], inp["k"], inp["v"], True, scale)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    g_ref = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], True, scale)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv), g_ref):
        check_grad(got, ref, name)
