"""GPU parity of the decode / short-query path (ffpa_decode_fwd) against the fp64 oracle.

The decode path computes the same forward as the tile kernels (FFPA docs,
"CuTe-DSL Backend" page, "Hard constraints": bottom-right causal, GQA/MQA,
empty rows give O = 0 and LSE = -inf) with the keys split over CTAs; these
tests cover one and several splits, ragged key tails, GQA groups that fill
the 16-row tile, causal rows with no legal key, strided views and no keys.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from head_dim_flash_gb300 import api
from head_dim_flash_gb300 import workloads
from tests.gpu_utils import Guarded, check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_dim_flash_gb300 import build

    build.build()
    oracle.build()


def run_decode(B, Hq, Hkv, Nq, Nkv, D, causal, dtype=torch.bfloat16, seed=0, amp=1.0, v_amp=None):
    inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, dtype, seed=seed, amplitude=amp)
    if v_amp is not None:
        # large logits from Q and K only: V stays unit-scale, so O's absolute
        # tolerance (a few bf16 half-ulps of unit values) still applies
        inp["v"] = (inp["v"].float() * (v_amp / amp)).to(dtype)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(D)
    og = Guarded(q.shape, dtype)
    lg = Guarded((B, Hq, Nq), torch.float32)
    assert api.decode_supported(q, k)
    api.decode_fwd(q, k, v, causal, scale, out=og.t, lse=lg.t)
    api.get_status()
    og.check_guards("o")
    lg.check_guards("lse")
    o_ref, lse_ref = oracle.attention_fwd(inp["q"], inp["k"], inp["v"], causal, scale)
    check_o(og.t, o_ref)
    check_lse(lg.t, lse_ref)
    empty = np.isneginf(lse_ref)
    if empty.any():
        o = og.t.float().cpu().numpy()
        assert np.all(o[empty] == 0.0)
        assert np.all(np.isneginf(lg.t.cpu().numpy()[empty]))
    return og.t, lg.t


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nkv", [(1, 1), (1, 100), (1, 4097), (3, 100), (7, 4097), (2, 33)])
def test_decode_mha_d512(Nq, Nkv, causal):
    run_decode(2, 4, 4, Nq, Nkv, 512, causal)


@pytest.mark.parametrize("G,Nq", [(4, 1), (8, 2), (16, 1), (4, 3)])
def test_decode_gqa_groups(G, Nq):
    run_decode(1, 2 * G, 2, Nq, 1500, 512, True)


@pytest.mark.parametrize("D", [64, 320, 576, 1024])
def test_decode_head_dims(D):
    run_decode(1, 8, 1, 1, 2000, D, False, seed=D)


def test_decode_fp16():
    run_decode(2, 8, 2, 1, 3000, 512, False, dtype=torch.float16, seed=5)


def test_decode_many_splits_long_context():
    # B * Hkv = 1: the keys spread over the largest split count
    run_decode(1, 8, 1, 2, 70000, 512, False, seed=9)


def test_decode_causal_rows_without_keys():
    # Nkv < Nq: bottom-right alignment leaves the first rows with no legal key
    run_decode(1, 2, 1, 8, 3, 512, True)


def test_decode_no_keys():
    run_decode(1, 4, 1, 2, 0, 512, False)


def test_decode_large_logits():
    run_decode(1, 8, 1, 1, 3000, 512, False, amp=4.0, seed=3, v_amp=1.0)


def test_decode_matches_tile_kernels():
    # same problem through both paths: both within tolerance of the oracle,
    # and close to each other
    inp = workloads.random_dense(2, 16, 2, 1, 5000, 512, torch.bfloat16, seed=11)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = api.decode_fwd(q, k, v, False, 0.05)
    o2, l2 = api.fwd(q, k, v, False, 0.05)
    api.get_status()
    torch.testing.assert_close(l1, l2, atol=1e-4, rtol=0)
    torch.testing.assert_close(o1.float(), o2.float(), atol=2e-2, rtol=2e-2)


def test_decode_strided_views():
    # q, k, v as [B, N, H, D] storage transposed to [B, H, N, D]; o into a
    # slice of a wider buffer
    B, Hq, Hkv, Nq, Nkv, D = 2, 8, 2, 2, 1000, 512
    inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, torch.bfloat16, seed=4)
    q = inp["q"].transpose(1, 2).contiguous().cuda().transpose(1, 2)
    k = inp["k"].transpose(1, 2).contiguous().cuda().transpose(1, 2)
    v = inp["v"].transpose(1, 2).contiguous().cuda().transpose(1, 2)
    wide = torch.full((B, Nq, Hq, D + 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = wide[..., :D].transpose(1, 2)
    _, lse = api.decode_fwd(q, k, v, True, 1.0 / math.sqrt(D), out=o)
    api.get_status()
    assert torch.isnan(wide[..., D:].float()).all()
    o_ref, lse_ref = oracle.attention_fwd(inp["q"], inp["k"], inp["v"], True, 1.0 / math.sqrt(D))
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("G,Nq,causal", [(32, 1, False), (8, 3, True), (4, 7, True), (1, 40, True)])
def test_decode_row_blocks(G, Nq, causal):
    # G * Nq > 16: several 16-row blocks per kv head, each reading K/V itself
    run_decode(1, 2 * G, 2, Nq, 777, 512, causal, seed=G + Nq)


def test_decode_rejects_unsupported_head_dim():
    q = torch.zeros(1, 4, 1, 352, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, 64, 352, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(NotImplementedError):
        api.decode_fwd(q, k, k, False, 0.05)


@pytest.mark.parametrize("Nq", [1, 5])
def test_attention_routes_short_queries_to_decode_with_gradients(Nq):
    # attention(): forward through the split-KV path for Nq < 8, backward
    # through the tile kernels; all against the oracle
    B, Hq, Hkv, Nkv, D = 1, 8, 2, 600, 512
    inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, torch.bfloat16, seed=Nq)
    q, k, v, do = (inp[n].cuda().requires_grad_(n != "dO") for n in ("q", "k", "v", "dO"))
    scale = 1.0 / math.sqrt(D)
    o = api.attention(q, k, v, True, scale)
    o.backward(do)
    api.get_status()
    o_ref, _ = oracle.attention_fwd(inp["q"], inp["k"], inp["v"], True, scale)
    check_o(o.detach(), o_ref)
    dq_ref, dk_ref, dv_ref = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], True, scale)
    check_grad(q.grad, dq_ref, "dQ")
    check_grad(k.grad, dk_ref, "dK")
    check_grad(v.grad, dv_ref, "dV")


def test_decode_full_size_workload():
    # the benchmarked decode workload, in the launch configuration the
    # benchmark times; every output against the oracle, one batch entry at a time
    w = workloads.DECODE
    inp = workloads.make_inputs(w, with_grad_out=False)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    og = Guarded(q.shape, w.dtype)
    lg = Guarded((w.B, w.Hq, w.Nq), torch.float32)
    api.decode_fwd(q, k, v, w.causal, w.scale, out=og.t, lse=lg.t)
    api.get_status()
    og.check_guards("o")
    lg.check_guards("lse")
    for b in range(w.B):
        o_ref, lse_ref = oracle.attention_fwd(inp["q"][b:b + 1], inp["k"][b:b + 1], inp["v"][b:b + 1], w.causal,
                                              w.scale)
        check_o(og.t[b:b + 1], o_ref, f"O[b{b}]")
        check_lse(lg.t[b:b + 1], lse_ref, f"LSE[b{b}]")
