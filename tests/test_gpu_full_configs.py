"""GPU parity at the five workloads' full sizes, in the launch configuration the
benchmark times (one ffpa_fwd and one ffpa_bwd call per workload).

The oracle cannot finish every head of the large workloads in seconds, so:
  * forward: sampled query rows of sampled heads are compared element by
    element (the oracle computes those rows exactly, one by one);
  * backward: whole heads (or whole GQA groups) are compared element by
    element, and two identities that hold for every head at any size are
    checked on ALL heads:  sum_j dK_j = 0  and  sum_j dV_j = sum over the
    group of the dO rows that have a legal key.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from head_dim_flash_gb300 import api
from head_dim_flash_gb300 import workloads as W
from tests.gpu_utils import check_grad, check_lse, check_o, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_dim_flash_gb300 import build

    build.build()
    oracle.build()


def run_gpu(w):
    inp = W.make_inputs(w)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "dO")}
    o, lse = api.fwd(dev["q"], dev["k"], dev["v"], w.causal, w.scale)
    dq, dk, dv = api.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], w.causal, w.scale)
    api.get_status()
    return inp, {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def sample_rows(n, k, seed):
    rng = np.random.default_rng(seed)
    rows = set([0, n - 1, n // 2]) | set(int(x) for x in rng.integers(0, n, k))
    return sorted(rows)


def check_forward_rows(inp, out, w, b, h, rows):
    hk = h // (w.Hq // w.Hkv)
    o_ref, lse_ref = oracle.attention_fwd_rows(inp["q"][b, h], inp["k"][b, hk], inp["v"][b, hk], rows, w.causal,
                                               w.scale)
    check_o(out["o"][b, h, rows], o_ref, f"O[b{b},h{h}]")
    check_lse(out["lse"][b, h, rows], lse_ref, f"LSE[b{b},h{h}]")


def check_group_backward(inp, out, w, b, hk):
    g = w.Hq // w.Hkv
    hs = slice(hk * g, (hk + 1) * g)
    sl = lambda t, s: t[b:b + 1, s]  # noqa: E731
    dq_ref, dk_ref, dv_ref = oracle.attention_bwd(sl(inp["q"], hs), sl(inp["k"], slice(hk, hk + 1)),
                                                  sl(inp["v"], slice(hk, hk + 1)), sl(inp["dO"], hs), w.causal,
                                                  w.scale)
    check_grad(sl(out["dq"], hs), dq_ref, f"dQ[b{b},group{hk}]")
    check_grad(sl(out["dk"], slice(hk, hk + 1)), dk_ref, f"dK[b{b},kv{hk}]")
    check_grad(sl(out["dv"], slice(hk, hk + 1)), dv_ref, f"dV[b{b},kv{hk}]")


def legal_rows_mask(nq, nk, causal):
    i = np.arange(nq)
    return (i + (nk - nq) >= 0) if causal else np.ones(nq, dtype=bool)


def check_invariants_all_heads(inp, out, w):
    """sum_j dK_j = 0 and sum_j dV_j = sum_{group, legal rows} dO_i, per (b, kv head)."""
    dk = out["dk"].double()
    dv = out["dv"].double()
    do = inp["dO"].double().cuda()
    g = w.Hq // w.Hkv
    mask = torch.as_tensor(legal_rows_mask(w.Nq, w.Nkv, w.causal), device=do.device)
    want_dv = (do * mask.view(1, 1, -1, 1)).sum(dim=2).view(w.B, w.Hkv, g, w.D).sum(dim=2)
    got_dk = dk.sum(dim=2)
    got_dv = dv.sum(dim=2)
    n = w.Nkv
    # bf16-rounded rows carry independent rounding errors: their sum drifts
    # like sqrt(n) * rms; a systematic error would drift like n * rms
    rms_dk = dk.pow(2).mean(dim=(2, 3)).sqrt()
    rms_dv = dv.pow(2).mean(dim=(2, 3)).sqrt()
    lim_dk = 0.05 * math.sqrt(n) * rms_dk.unsqueeze(-1)
    lim_dv = 0.05 * math.sqrt(n) * rms_dv.unsqueeze(-1)
    assert torch.all(got_dk.abs() <= lim_dk), float((got_dk.abs() / lim_dk).max())
    assert torch.all((got_dv - want_dv).abs() <= lim_dv), float(((got_dv - want_dv).abs() / lim_dv).max())


def test_headline_dense_b1_h32_n8192_d512():
    w = W.HEADLINE
    inp, out = run_gpu(w)
    for h in (0, 17, 31):
        check_forward_rows(inp, out, w, 0, h, sample_rows(w.Nq, 40, h))
    check_invariants_all_heads(inp, out, w)
    check_group_backward(inp, out, w, 0, 17)


def test_causal_gqa_cross_b2_hq32_hkv8_nq4096_nkv8192():
    w = W.GQA_CAUSAL
    inp, out = run_gpu(w)
    for b, hs in ((0, (0, 3)), (1, (28, 31))):
        for h in hs:
            check_forward_rows(inp, out, w, b, h, sample_rows(w.Nq, 40, 100 + h))
    check_invariants_all_heads(inp, out, w)
    check_group_backward(inp, out, w, 0, 0)


@pytest.mark.parametrize("idx", [0, 1, 2], ids=["D320", "D640", "D1024"])
def test_head_dim_sweep_fp16_n4000(idx):
    w = W.SWEEP[idx]
    inp, out = run_gpu(w)
    for h in (0, 15):
        check_forward_rows(inp, out, w, 0, h, sample_rows(w.Nq, 40, h))
    check_invariants_all_heads(inp, out, w)
    check_group_backward(inp, out, w, 0, 0)


def test_varlen_packed_six_sequences_causal():
    w = W.VARLEN
    inp = W.make_inputs(w)
    cu = inp["cu_seqlens"]
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "dO")}
    cuq = cu.cuda()
    mx = max(w.seqlens)
    o, lse = api.varlen_fwd(dev["q"], dev["k"], dev["v"], cuq, cuq, mx, mx, True, w.scale)
    dq, dk, dv = api.varlen_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], cuq, cuq, mx, mx, True, w.scale)
    api.get_status()
    # forward: heads {0, 31} of every sequence, all rows
    heads = [0, 31]
    o_ref, lse_ref = oracle.varlen_fwd(inp["q"][:, heads], inp["k"][:, heads], inp["v"][:, heads], cu, cu, True,
                                       w.scale)
    check_o(o[:, heads], o_ref)
    check_lse(lse[heads], lse_ref)
    # backward: head 0 of every sequence, all rows and keys
    g_ref = oracle.varlen_bwd(inp["q"][:, :1], inp["k"][:, :1], inp["v"][:, :1], inp["dO"][:, :1], cu, cu, True,
                              w.scale)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dq[:, :1], dk[:, :1], dv[:, :1]), g_ref):
        check_grad(got, ref, name)
    # identities on every head of every sequence
    for bi in range(len(w.seqlens)):
        s, e = int(cu[bi]), int(cu[bi + 1])
        dks = to64(dk[s:e]).sum(axis=0)
        rms = np.sqrt((to64(dk[s:e]) ** 2).mean(axis=(0, 2)))
        assert np.all(np.abs(dks) <= 0.05 * math.sqrt(e - s) * rms[:, None])
