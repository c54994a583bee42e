"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Small and ragged shapes are compared element by element on every output,
with NaN-prefilled outputs and canaries around every buffer. The tolerances
live in tests/gpu_utils.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from head_dim_flash_gb300 import api
from head_dim_flash_gb300 import workloads
from tests.gpu_utils import Guarded, check_empty_rows_exact, check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_dim_flash_gb300 import build

    build.build()
    oracle.build()


def run_dense(B, Hq, Hkv, Nq, Nkv, D, causal, dtype=torch.bfloat16, seed=0, amp=1.0, scale=None, backward=True,
              v_amp=None):
    inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, dtype, seed=seed, amplitude=amp)
    if v_amp is not None:
        inp["v"] = (inp["v"].float() * (v_amp / amp)).to(dtype)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    og = Guarded(q.shape, dtype)
    lg = Guarded((B, Hq, Nq), torch.float32)
    api.fwd(q, k, v, causal, scale, out=og.t, lse=lg.t)
    api.get_status()
    og.check_guards("o")
    lg.check_guards("lse")
    o_ref, lse_ref = oracle.attention_fwd(inp["q"], inp["k"], inp["v"], causal, scale)
    check_o(og.t, o_ref)
    check_lse(lg.t, lse_ref)
    if not backward:
        return
    dqg, dkg, dvg = Guarded(q.shape, dtype), Guarded(k.shape, dtype), Guarded(v.shape, dtype)
    api.bwd(q, k, v, og.t, lg.t, do, causal, scale, dq=dqg.t, dk=dkg.t, dv=dvg.t)
    api.get_status()
    for name, gd in (("dq", dqg), ("dk", dkg), ("dv", dvg)):
        gd.check_guards(name)
    dq_ref, dk_ref, dv_ref = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], causal, scale)
    check_grad(dqg.t, dq_ref, "dQ")
    check_grad(dkg.t, dk_ref, "dK")
    check_grad(dvg.t, dv_ref, "dV")
    empty = np.isneginf(lse_ref)
    if empty.any():
        check_empty_rows_exact(og.t, lg.t, dqg.t, empty)


def test_tiny_config_full_parity():
    w = workloads.TINY
    inp = workloads.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    o, lse = api.fwd(q, k, v, w.causal, w.scale)
    dq, dk, dv = api.bwd(q, k, v, o, lse, do, w.causal, w.scale)
    api.get_status()
    o_ref, lse_ref = oracle.attention_fwd(inp["q"], inp["k"], inp["v"], w.causal, w.scale)
    g_ref = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], w.causal, w.scale)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv), g_ref):
        check_grad(got, ref, name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 128, 129, 300])
def test_ragged_lengths_d512(N, causal):
    run_dense(1, 2, 2, N, N, 512, causal, seed=N)


@pytest.mark.parametrize("D", [64, 128, 320, 640, 1024])
def test_head_dims(D):
    run_dense(1, 2, 1, 200, 260, D, False, dtype=torch.float16, seed=D, amp=0.5)


@pytest.mark.parametrize("D,causal,dtype", [(96, False, torch.float16), (160, True, torch.bfloat16),
                                             (352, True, torch.float16), (736, False, torch.bfloat16)])
def test_head_dims_multiple_of_32(D, causal, dtype):
    # D % 64 = 32: the last 64-wide chunk is half zero fill
    run_dense(1, 4, 2, 200, 260, D, causal, dtype=dtype, seed=D + 1, amp=0.5)


@pytest.mark.parametrize("causal", [False, True])
def test_cross_attention_gqa(causal):
    # Nq < Nkv bottom-right causal with a 4-way GQA group
    run_dense(2, 8, 2, 150, 333, 512, causal, seed=11)


def test_causal_more_queries_than_keys_gives_empty_rows():
    # Nq > Nkv: rows 0..Nq-Nkv-1 have no legal key: O=0, LSE=-inf, zero dQ
    run_dense(1, 2, 1, 300, 100, 512, True, seed=12)


def test_fp16_causal_gqa():
    run_dense(1, 4, 1, 257, 257, 320, True, dtype=torch.float16, seed=13, amp=0.5)


@pytest.mark.parametrize("causal", [False, True])
def test_large_scores_trigger_rescaling(causal):
    # q, k amplitude 3 and scale 1: scores of magnitude ~100 make the running
    # row max jump by far more than 2^8 between key tiles, exercising the lazy
    # O rescale; v keeps amplitude 1 so |O| stays where bf16 resolves 2e-2
    run_dense(1, 2, 1, 256, 1024, 128, causal, seed=14, amp=3.0, scale=1.0, v_amp=1.0)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_oracle(causal):
    lq = [5, 0, 130, 257, 64]
    lk = [7, 3, 130, 200, 0]
    inp = workloads.random_varlen(lq, lk, 4, 2, 512, seed=21)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    cq, ck = inp["cu_seqlens_q"].cuda(), inp["cu_seqlens_k"].cuda()
    scale = 1 / math.sqrt(512)
    o, lse = api.varlen_fwd(q, k, v, cq, ck, max(lq), max(lk), causal, scale)
    dq, dk, dv = api.varlen_bwd(q, k, v, o, lse, do, cq, ck, max(lq), max(lk), causal, scale)
    api.get_status()
    o_ref, lse_ref = oracle.varlen_fwd(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                                       causal, scale)
    g_ref = oracle.varlen_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                              causal, scale)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv), g_ref):
        check_grad(got, ref, name)


# Both kernel families (one CTA per head-dim slab; CTA pairs with 2-SM MMAs)
# on shapes the automatic choice by head dim would not give them.
@pytest.mark.parametrize("family", ["single", "pair"])
@pytest.mark.parametrize("D,causal", [(512, True), (64, False), (320, True), (1024, False)])
def test_kernel_families(family, D, causal, monkeypatch):
    monkeypatch.setenv("FFPA_KERNEL", family)
    run_dense(1, 4, 2, 150, 333, D, causal, dtype=torch.float16, seed=40 + D, amp=0.5)


@pytest.mark.parametrize("family", ["single", "pair"])
def test_kernel_families_varlen_causal(family, monkeypatch):
    monkeypatch.setenv("FFPA_KERNEL", family)
    lq = [130, 1, 300]
    lk = [200, 5, 260]
    inp = workloads.random_varlen(lq, lk, 2, 1, 512, seed=45)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    cq, ck = inp["cu_seqlens_q"].cuda(), inp["cu_seqlens_k"].cuda()
    scale = 1 / math.sqrt(512)
    o, lse = api.varlen_fwd(q, k, v, cq, ck, max(lq), max(lk), True, scale)
    dq, dk, dv = api.varlen_bwd(q, k, v, o, lse, do, cq, ck, max(lq), max(lk), True, scale)
    api.get_status()
    o_ref, lse_ref = oracle.varlen_fwd(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                                       True, scale)
    g_ref = oracle.varlen_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                              True, scale)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv), g_ref):
        check_grad(got, ref, name)


def test_autograd_entry_points():
    inp = workloads.random_dense(1, 2, 2, 64, 64, 512, torch.bfloat16, seed=31)
    q, k, v = (inp[n].cuda().requires_grad_(True) for n in ("q", "k", "v"))
    from head_dim_flash_gb300 import api as attn_mod

    o = attn_mod.attention(q, k, v, causal=True)
    o.backward(inp["dO"].cuda())
    g_ref = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], True, 1 / math.sqrt(512))
    for name, got, ref in zip(("dQ", "dK", "dV"), (q.grad, k.grad, v.grad), g_ref):
        check_grad(got, ref, name)


def test_bounded_wait_reports_timeout():
    from head_dim_flash_gb300 import _ffi

    st = _ffi.ffpa_selftest_wait_timeout(20_000_000, torch.cuda.current_stream().cuda_stream)
    assert st == _ffi.ERR_TIMEOUT
    # the context stays usable and the status word is cleared
    assert _ffi.ffpa_get_status(torch.cuda.current_stream().cuda_stream) == _ffi.OK
    run_dense(1, 1, 1, 64, 64, 128, False, backward=False)
