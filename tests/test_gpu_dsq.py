"""GPU parity of the stored-dS backward: the dK launch also writes dS^T to the
workspace and dQ = scale dS K is one GEMM (dense, D = 256 / 512, causal or not).

Every case runs the backward twice on the same inputs, with the small
workspace (dQ recomputes S and dP) and with the stored-dS workspace, and
checks both against the fp64 oracle with the usual gradient tolerance; dV (and
dK when non-causal) must be bit-identical between the two.
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


def run_both(B, Hq, Hkv, Nq, Nkv, D, dtype=torch.bfloat16, seed=0, causal=False):
    inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, dtype, seed=seed)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    scale = 1.0 / math.sqrt(D)
    o, lse = api.fwd(q, k, v, causal, scale)
    small = torch.empty(api.bwd_workspace_bytes(q, k), dtype=torch.uint8, device="cuda")
    big_n = api.bwd_workspace_bytes(q, k, causal)
    assert big_n > small.numel(), "the stored-dS path applies to this problem"
    big = torch.empty(big_n, dtype=torch.uint8, device="cuda")
    g_small = api.bwd(q, k, v, o, lse, do, causal, scale, workspace=small)
    g_big = api.bwd(q, k, v, o, lse, do, causal, scale, workspace=big)
    api.get_status()
    ref = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], causal, scale)
    for gs in (g_small, g_big):
        for name, got, r in zip(("dQ", "dK", "dV"), gs, ref):
            check_grad(got, r, name)
    # dV is the same kernel either way; dK too, except that causal storing starts
    # at an even query tile (an extra all-masked tile shifts its summation order)
    assert torch.equal(g_small[2], g_big[2])
    if not causal:
        assert torch.equal(g_small[1], g_big[1])
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


@pytest.mark.parametrize("Nq,Nkv", [(300, 300), (256, 700), (700, 256), (100, 1000), (513, 769)])
def test_stored_ds_backward_causal(Nq, Nkv):
    # bottom-right causal: the dQ GEMM stops at each tile's last legal key, and
    # rows with no legal key (Nq > Nkv) get dQ = 0
    run_both(1, 4, 2, Nq, Nkv, 512, seed=Nq + 2 * Nkv, causal=True)


def test_varlen_and_other_head_dims_keep_the_recompute_path():
    q = torch.zeros(1, 2, 64, 320, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 2, 64, 320, dtype=torch.bfloat16, device="cuda")
    assert api.bwd_workspace_bytes(q, k, True) == api.bwd_workspace_bytes(q, k)
    q5 = torch.zeros(1, 2, 64, 512, dtype=torch.bfloat16, device="cuda")
    assert api.bwd_workspace_bytes(q5, q5, True) > api.bwd_workspace_bytes(q5, q5)


def test_one_cta_family_forced_keeps_the_recompute_path(monkeypatch):
    # only the CTA-pair dK kernel stores dS: with the one-CTA family forced, the
    # large workspace must still give the recompute path's (correct) dQ
    monkeypatch.setenv("FFPA_KERNEL", "single")
    run_both(1, 4, 2, 150, 333, 512, dtype=torch.float16, seed=552, causal=True)
