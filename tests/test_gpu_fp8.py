"""GPU parity of the FP8 (e4m3) forward against the oracle's FP8 reference.

* Quantization: the e4m3 codes of Q, K and V (V transposed) and the fp32
  per-(batch, head) scales are compared bit for bit (+0 and -0 count as the
  same code).
* Forward: O against the plain attention of the dequantized inputs (fp64),
  element by element within
      bound (the e4m3 rounding of P, oracle.fp8.p_rounding_bound)
      + 2^-8 |O| (rounding of the 16-bit output)
      + 1e-3 max|V| (a margin, not a derived bound: it stands for the
        rounding of the score and P.V accumulations and of exp2, which the
        P bound leaves out; the tensor cores' accumulation order and internal
        precision for e4m3 operands are not publicly documented, so no bound
        is derived for them),
  and LSE within 1e-3.
* Head dims: every multiple of 32 in [64, 1024] (the pages' FP8 range); the
  codes are padded to a multiple of 128 head-dim columns with zero codes,
  which the quantization pass writes and the tests check.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
from head_dim_flash_gb300 import api
from head_dim_flash_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_dim_flash_gb300 import build

    build.build()
    oracle.build()


def same_codes(got, ref):
    got = np.asarray(got, dtype=np.uint8)
    ref = np.asarray(ref, dtype=np.uint8)
    both_zero = ((got & 0x7F) == 0) & ((ref & 0x7F) == 0)
    return np.all((got == ref) | both_zero)


def check_quantization(inp, q, k, v):
    _, views = api.fp8_quantize(q, k, v)
    torch.cuda.synchronize()
    for name, src in (("q", inp["q"]), ("k", inp["k"]), ("v", inp["v"])):
        codes, scale = ofp8.quantize(src)
        got_s = views["s" + name].cpu().numpy()
        assert np.array_equal(got_s, scale), f"{name}: scales differ"
        if name == "v":
            n = codes.shape[2]
            got = views["v8t"].cpu().numpy()[..., :n]
            ref = codes.transpose(0, 1, 3, 2)
        else:
            got = views[name + "8"].cpu().numpy()
            ref = codes
        assert same_codes(got, ref), f"{name}: {int((got != ref).sum())} codes differ"
    # the head-dim pad past D holds zero codes (q, k: columns; V^T: rows)
    D = q.shape[3]
    assert not views["q8_padded"][..., D:].any() and not views["k8_padded"][..., D:].any()
    assert not views["v8t_padded"][:, :, D:].any()


def run_fp8(B, Hq, Hkv, Nq, Nkv, D, causal, dtype=torch.bfloat16, seed=0, amp=1.0, strided=False):
    inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, dtype, seed=seed, amplitude=amp, with_grad_out=False)
    if strided:
        # [B, N, H, D] storage seen as [B, H, N, D]
        q, k, v = (inp[n].transpose(1, 2).contiguous().cuda().transpose(1, 2) for n in ("q", "k", "v"))
    else:
        q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(D)
    check_quantization(inp, q, k, v)
    o, lse = api.fwd_fp8(q, k, v, causal, scale)
    api.get_status()
    o_ref, lse_ref, (qd, kd, vd) = ofp8.attention_fwd_fp8(inp["q"], inp["k"], inp["v"], causal, scale)
    bound = ofp8.p_rounding_bound(qd, kd, vd, causal, scale)
    og = o.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(og))
    vmax = np.abs(vd).max()
    tol = bound + 2.0 ** -8 * np.abs(o_ref) + 1e-3 * vmax
    err = np.abs(og - o_ref)
    ratio = float((err / tol).max())
    assert np.all(err <= tol), f"O: max err {err.max():.3e}, max err/tol {ratio:.3f}"
    lg = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    assert np.all(np.abs(lg[fin] - lse_ref[fin]) <= 1e-3), f"LSE max err {np.abs(lg[fin] - lse_ref[fin]).max():.3e}"
    return ratio


@pytest.mark.parametrize("D", [64, 96, 128, 256, 320, 384, 512, 640, 768, 896, 1024])
def test_fp8_head_dims(D):
    run_fp8(1, 2, 2, 300, 300, D, False, seed=D)


@pytest.mark.parametrize("D", [160, 448, 1024])
def test_fp8_head_dims_causal_gqa(D):
    run_fp8(1, 4, 2, 257, 400, D, True, seed=D + 1)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nkv", [(1, 129), (256, 256), (257, 1000), (700, 333)])
def test_fp8_ragged_and_causal(Nq, Nkv, causal):
    run_fp8(1, 2, 1, Nq, Nkv, 512, causal, seed=Nq + Nkv)


def test_fp8_d768_causal_gqa():
    run_fp8(1, 6, 2, 300, 520, 768, True, seed=17)


def test_fp8_gqa_fp16():
    run_fp8(2, 8, 2, 200, 700, 512, True, dtype=torch.float16, seed=7, amp=0.5)


def test_fp8_large_logits():
    run_fp8(1, 2, 2, 256, 512, 512, False, seed=8, amp=3.0)


def test_fp8_strided_views():
    run_fp8(2, 4, 2, 130, 260, 512, False, seed=9, strided=True)


def test_fp8_prequantized_matches_one_call():
    # quantize once, attend from the workspace: bit-identical to ffpa_fwd_fp8
    inp = workloads.random_dense(1, 4, 2, 200, 333, 512, torch.bfloat16, seed=12, with_grad_out=False)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = api.fwd_fp8(q, k, v, True, 0.05)
    ws, _ = api.fp8_quantize(q, k, v)
    o2, l2 = api.fwd_fp8_quantized(ws, q.shape, k.shape, q.dtype, True, 0.05)
    api.get_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fp8_full_size_workload_sampled():
    # the benchmarked FP8 workload in the benchmark's launch configuration:
    # codes of sampled heads bit for bit, sampled query rows of those heads
    # against the oracle within the bound (rows are independent: non-causal)
    w = workloads.FP8
    inp = workloads.make_inputs(w, with_grad_out=False)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    ws = api.fp8_workspace(q, k)
    o, lse = api.fwd_fp8(q, k, v, w.causal, w.scale, workspace=ws)
    api.get_status()
    _, views = api.fp8_quantize(q, k, v, workspace=ws)
    rng = np.random.default_rng(0)
    for h in (0, 17, 31):
        sl = slice(h, h + 1)
        cq, sq = ofp8.quantize(inp["q"][:, sl])
        ck, sk = ofp8.quantize(inp["k"][:, sl])
        cv, sv = ofp8.quantize(inp["v"][:, sl])
        assert same_codes(views["q8"][:, sl].cpu().numpy(), cq)
        assert same_codes(views["k8"][:, sl].cpu().numpy(), ck)
        assert same_codes(views["v8t"][:, sl, :, : w.Nkv].cpu().numpy(), cv.transpose(0, 1, 3, 2))
        assert views["sq"][0, h].item() == sq[0, 0] and views["sv"][0, h].item() == sv[0, 0]
        qd, kd, vd = ofp8.dequantize(cq, sq), ofp8.dequantize(ck, sk), ofp8.dequantize(cv, sv)
        rows = sorted(set([0, w.Nq - 1]) | set(int(x) for x in rng.integers(0, w.Nq, 24)))
        o_ref, lse_ref = oracle.attention_fwd_rows(qd[0, 0], kd[0, 0], vd[0, 0], rows, False, w.scale)
        bound = ofp8.p_rounding_bound(qd[:, :, rows], kd, vd, False, w.scale)[0, 0]
        og = o[0, h, rows].float().cpu().numpy().astype(np.float64)
        tol = bound + 2.0 ** -8 * np.abs(o_ref) + 1e-3 * np.abs(vd).max()
        assert np.all(np.abs(og - o_ref) <= tol), f"head {h}: max err {np.abs(og - o_ref).max():.3e}"
        assert np.all(np.abs(lse[0, h, rows].cpu().numpy() - lse_ref) <= 1e-3)


def test_fp8_all_zero_heads():
    # an all-zero K head (scale 1, zero codes: uniform weights) and an all-zero V head
    inp = workloads.random_dense(1, 4, 2, 130, 260, 512, torch.bfloat16, seed=21, with_grad_out=False)
    inp["k"][:, 0] = 0
    inp["v"][:, 1] = 0
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    check_quantization(inp, q, k, v)
    o, lse = api.fwd_fp8(q, k, v, False, 0.05)
    api.get_status()
    o_ref, lse_ref, (qd, kd, vd) = ofp8.attention_fwd_fp8(inp["q"], inp["k"], inp["v"], False, 0.05)
    tol = ofp8.p_rounding_bound(qd, kd, vd, False, 0.05) + 2.0 ** -8 * np.abs(o_ref) + 1e-3 * np.abs(vd).max()
    assert np.all(np.abs(o.float().cpu().numpy() - o_ref) <= tol)
    assert np.all(o[:, 2:4].float().cpu().numpy() == 0.0)   # heads of the zero V head
    assert np.all(np.abs(lse.cpu().numpy() - lse_ref) <= 1e-3)


def run_fp8_varlen(lq, lk, Hq, Hkv, D, causal, dtype=torch.bfloat16, seed=0):
    """Packed FP8 forward against the oracle's per-sequence FP8 reference, with
    the tolerance of run_fp8 (derived P-rounding bound per sequence, output
    rounding, the stated margin)."""
    inp = workloads.random_varlen(lq, lk, Hq, Hkv, D, dtype, seed=seed)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    cq, ck = inp["cu_seqlens_q"], inp["cu_seqlens_k"]
    scale = 1.0 / math.sqrt(D)
    o, lse = api.varlen_fwd_fp8(q, k, v, cq.cuda(), ck.cuda(), max(lq), max(lk), causal, scale)
    api.get_status()
    o_ref, lse_ref, bound = ofp8.varlen_attention_fwd_fp8(inp["q"], inp["k"], inp["v"], cq.numpy(), ck.numpy(),
                                                          causal, scale)
    og = o.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(og))
    vmax = float(np.abs(inp["v"].float().numpy()).max())
    tol = bound + 2.0 ** -8 * np.abs(o_ref) + 1e-3 * vmax
    err = np.abs(og - o_ref)
    assert np.all(err <= tol), f"O: max err {err.max():.3e}, max err/tol {float((err / tol).max()):.3f}"
    lg = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    assert np.all(np.abs(lg[fin] - lse_ref[fin]) <= 1e-3), f"LSE max err {np.abs(lg[fin] - lse_ref[fin]).max():.3e}"


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_varlen_d512(causal):
    # ragged lengths (several row and key tiles, tails), a zero-length query
    # sequence, and a sequence whose keys start off a 16-column boundary
    run_fp8_varlen([300, 0, 129, 517], [300, 37, 400, 517], 4, 2, 512, causal, seed=21)


@pytest.mark.parametrize("D", [64, 96, 320, 1024])
def test_fp8_varlen_head_dims(D):
    run_fp8_varlen([70, 200, 33], [150, 5, 260], 2, 2, D, True, seed=D + 3)


def test_fp8_varlen_keyless_sequence_and_fp16():
    # a sequence without keys gives O = 0, LSE = -inf
    run_fp8_varlen([40, 90, 17], [0, 300, 64], 8, 2, 512, False, dtype=torch.float16, seed=33)


def test_fp8_varlen_bound_below_longest_sequence_is_an_error():
    inp = workloads.random_varlen([100, 300], [100, 300], 2, 2, 512, torch.bfloat16, seed=5)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    cq, ck = inp["cu_seqlens_q"].cuda(), inp["cu_seqlens_k"].cuda()
    api.varlen_fwd_fp8(q, k, v, cq, ck, 299, 300, False, 0.05)
    with pytest.raises(ValueError, match="varlen contract"):
        api.get_status()
