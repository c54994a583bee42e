"""GPU parity of the stored-dS backward: the dK launch also writes dS^T to the
workspace and dQ = scale dS K is one GEMM (dense, non-causal, D = 256 / 512).

Every case runs the backward twice on the same inputs, with the small
workspace (dQ recomputes S and dP) and with the stored-dS workspace, and
checks both against the fp64 oracle with the usual gradient tolerance; dK and
dV must be bit-identical between the two (the same kernels compute them).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from head_dim_flash_gb300 import api
from head_dim_flash_gb300 import workloads
from tests.gpu_utils import check_grad

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_dim_flash_gb300 import build

    build.build()
    oracle.build()


def run_both(B, Hq, Hkv, Nq, Nkv, D, dtype=torch.bfloat16, seed=0):
    inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, dtype, seed=seed)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    scale = 1.0 / math.sqrt(D)
    o, lse = api.fwd(q, k, v, False, scale)
    small = torch.empty(api.bwd_workspace_bytes(q, k), dtype=torch.uint8, device="cuda")
    big_n = api.bwd_workspace_bytes(q, k, False)
    assert big_n > small.numel(), "the stored-dS path applies to this problem"
    big = torch.empty(big_n, dtype=torch.uint8, device="cuda")
    g_small = api.bwd(q, k, v, o, lse, do, False, scale, workspace=small)
    g_big = api.bwd(q, k, v, o, lse, do, False, scale, workspace=big)
    api.get_status()
    ref = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], False, scale)
    for gs in (g_small, g_big):
        for name, got, r in zip(("dQ", "dK", "dV"), gs, ref):
            check_grad(got, r, name)
    assert torch.equal(g_small[1], g_big[1]) and torch.equal(g_small[2], g_big[2])
    return inp, (q, k, v, do, o, lse, scale, big), g_big


@pytest.mark.parametrize("D", [256, 512])
@pytest.mark.parametrize("Nq,Nkv", [(256, 256), (301, 333), (1000, 129), (64, 700)])
def test_stored_ds_backward(D, Nq, Nkv):
    run_both(1, 2, 2, Nq, Nkv, D, seed=Nq + D)


def test_stored_ds_backward_gqa_fp16():
    run_both(2, 8, 2, 300, 520, 512, dtype=torch.float16, seed=3)


def test_stage_bit_4_replays_the_gemm_on_the_stored_ds():
    # preprocess, dK (stores dS), then bit 4 alone: the same dQ as the full call
    inp, (q, k, v, do, o, lse, scale, big), (dq_full, _, _) = run_both(1, 4, 2, 512, 512, 512, seed=5)
    dq = torch.empty_like(q)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    for bit in (1, 8, 16):
        api.bwd(q, k, v, o, lse, do, False, scale, workspace=big, dq=dq, dk=dk, dv=dv, stages=bit)
    api.get_status()
    assert torch.equal(dq, dq_full)


def test_causal_problems_keep_the_recompute_path():
    q = torch.zeros(1, 2, 64, 512, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 2, 64, 512, dtype=torch.bfloat16, device="cuda")
    assert api.bwd_workspace_bytes(q, k, True) == api.bwd_workspace_bytes(q, k)
    assert api.bwd_workspace_bytes(q, k, False) > api.bwd_workspace_bytes(q, k)
