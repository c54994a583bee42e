"""GPU tests of the launch limits and of the device-side varlen contract check.

- The packed varlen entry points read cu_seqlens on the device. A sequence
  longer than max_seqlen_q / max_seqlen_k (which size the launch), or offsets
  that run past the packed totals, must come back as FFPA_ERR_INVALID_VALUE
  from the status word (ValueError in Python), not as a silently partial
  result (FFPA docs, "CuTe-DSL Backend" page, "Varlen (packed THD) API": an
  actionable error instead of silently unpacking). The check only writes a
  status word; the kernels return normally and the context stays usable.
- More than 65535 (batch, head) pairs in one call: the launch grids spread
  the work units over two grid dimensions ("CuTe-DSL Backend" page, "Hard
  constraints", lists no limit on B * H). Checked against the fp64 oracle.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from head_dim_flash_gb300 import api, workloads
from tests.gpu_utils import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


def _varlen_inputs(D=512, seed=61):
    lq = [130, 300, 17]
    lk = [200, 260, 40]
    inp = workloads.random_varlen(lq, lk, 2, 1, D, seed=seed)
    return lq, lk, inp


@pytest.mark.parametrize("family,D", [("pair", 512), ("single", 320)])
@pytest.mark.parametrize("side", ["q", "k"])
def test_varlen_bound_below_longest_sequence_is_an_error(family, D, side, monkeypatch):
    monkeypatch.setenv("FFPA_KERNEL", family)
    lq, lk, inp = _varlen_inputs(D)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    cq, ck = inp["cu_seqlens_q"].cuda(), inp["cu_seqlens_k"].cuda()
    scale = 1 / math.sqrt(D)
    mq, mk = max(lq), max(lk)
    bad_q, bad_k = (mq - 1, mk) if side == "q" else (mq, mk - 1)
    # forward with a bound one below the longest sequence: an error, not a partial result
    api.varlen_fwd(q, k, v, cq, ck, bad_q, bad_k, True, scale)
    with pytest.raises(ValueError, match="varlen contract"):
        api.get_status()
    # the status word was cleared and the context is usable: the same call with
    # the true bounds matches the oracle
    o, lse = api.varlen_fwd(q, k, v, cq, ck, mq, mk, True, scale)
    api.get_status()
    o_ref, lse_ref = oracle.varlen_fwd(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                                       True, scale)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    # backward (stored-tile path where it applies, else recompute) with the bad bound
    api.varlen_bwd(q, k, v, o, lse, do, cq, ck, bad_q, bad_k, True, scale)
    with pytest.raises(ValueError, match="varlen contract"):
        api.get_status()
    dq, dk, dv = api.varlen_bwd(q, k, v, o, lse, do, cq, ck, mq, mk, True, scale)
    api.get_status()
    g_ref = oracle.varlen_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                              True, scale)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv), g_ref):
        check_grad(got, ref, name)


def test_varlen_offsets_past_total_are_an_error():
    lq, lk, inp = _varlen_inputs()
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    cq = inp["cu_seqlens_q"].clone()
    cq[-1] += 8  # the last sequence runs 8 tokens past total_q
    scale = 1 / math.sqrt(512)
    api.varlen_fwd(q, k, v, cq.cuda(), inp["cu_seqlens_k"].cuda(), max(lq) + 8, max(lk), False, scale)
    with pytest.raises(ValueError, match="sequence 2"):
        api.get_status()


def _dense(B, Hq, Hkv, Nq, Nkv, D, seed, causal):
    inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, torch.bfloat16, seed=seed)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    scale = 1 / math.sqrt(D)
    o, lse = api.fwd(q, k, v, causal, scale)
    dq, dk, dv = api.bwd(q, k, v, o, lse, do, causal, scale)
    api.get_status()
    o_ref, lse_ref = oracle.attention_fwd(inp["q"], inp["k"], inp["v"], causal, scale)
    g_ref = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], causal, scale)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv), g_ref):
        check_grad(got, ref, name)


# 70000 (batch, head) pairs: more work units than one grid dimension holds,
# for the one-CTA family (D = 64), the CTA-pair family (D = 256) and GQA
@pytest.mark.parametrize("B,Hq,Hkv,D,causal", [(70000, 1, 1, 64, False), (35000, 2, 2, 256, True),
                                                (17500, 4, 2, 64, True)])
def test_more_than_65535_heads(B, Hq, Hkv, D, causal):
    _dense(B, Hq, Hkv, 3, 5, D, seed=70 + D, causal=causal)


def test_decode_more_than_65535_units():
    inp = workloads.random_dense(70000, 1, 1, 1, 40, 64, torch.bfloat16, seed=77, with_grad_out=False)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    scale = 1 / math.sqrt(64)
    o, lse = api.decode_fwd(q, k, v, False, scale)
    api.get_status()
    o_ref, lse_ref = oracle.attention_fwd(inp["q"], inp["k"], inp["v"], False, scale)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def test_fp8_quantization_more_than_65535_heads():
    from oracle import fp8 as ofp8
    from tests.test_gpu_fp8 import same_codes

    B = 22000  # 66000 heads of q, k and v in the quantization grids
    inp = workloads.random_dense(B, 1, 1, 2, 3, 256, torch.bfloat16, seed=78, with_grad_out=False)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    _, views = api.fp8_quantize(q, k, v)
    torch.cuda.synchronize()
    api.get_status()
    # bit-exact codes and scales for a sample of batch entries at both ends
    for sl in (slice(0, 3), slice(B - 3, B)):
        for name, src in (("q", inp["q"]), ("k", inp["k"])):
            codes, scales = ofp8.quantize(src[sl])
            assert same_codes(views[name + "8"][sl].cpu().numpy(), codes), name
            np.testing.assert_array_equal(views["s" + name][sl].cpu().numpy(), scales)
