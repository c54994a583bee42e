"""Pins of the FP8 (e4m3) reference in oracle/fp8.py, independent of it.

* e4m3 rounding against torch's float8_e4m3fn cast (a library routine) over
  the representable range, and an exhaustive round trip of all 256 codes;
* ties to even, saturation and subnormals from the format's definition
  (values written out by hand);
* per-head quantization invariants (the amax element maps to +-448, the
  error of a dequantized value is at most half a unit in its last place);
* the P-rounding error bound, checked by brute force: P rounded to e4m3
  relative to the exact row maximum and to stale maxima up to 8 (log2 units)
  below it, the rounded O never leaves the bound.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def test_round_matches_torch_float8_cast():
    rng = np.random.default_rng(0)
    y = np.concatenate([
        rng.standard_normal(20000) * 30.0,
        rng.uniform(-448.0, 448.0, 20000),
        rng.standard_normal(20000) * 2.0 ** -7,      # subnormal range
        rng.standard_normal(2000) * 2.0 ** -11,      # below the smallest subnormal
    ]).astype(np.float32)
    y = y[np.abs(y) <= 448.0]
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.e4m3_round(y)
    assert np.array_equal(np.abs(got), np.abs(ref))
    nz = ref != 0
    assert np.array_equal(np.sign(got[nz]), np.sign(ref[nz]))


def test_all_codes_round_trip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = fp8.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(vals, ref)
    assert np.array_equal(fp8.e4m3_round(vals), vals)
    assert np.array_equal(fp8.e4m3_encode(vals), codes)


def test_ties_saturation_and_subnormals():
    # 1 + 1/16 lies halfway between 1 and 1.125: ties to the even mantissa (1)
    # 1 + 3/16 lies halfway between 1.125 and 1.25: ties to 1.25 (mantissa 010)
    assert fp8.e4m3_round([1.0625, 1.1875]).tolist() == [1.0, 1.25]
    assert fp8.e4m3_round([448.0, 460.0, 1e6, -1e9]).tolist() == [448.0, 448.0, 448.0, -448.0]
    # subnormals are multiples of 2^-9; half of the smallest one rounds to 0 (tie to even)
    s = 2.0 ** -9
    assert fp8.e4m3_round([s, 1.5 * s, 0.5 * s, 0.51 * s, 7 * s, 7.5 * s]).tolist() == [s, 2 * s, 0.0, s, 7 * s, 8 * s]
    assert fp8.e4m3_encode([448.0, -448.0, 2.0 ** -6, s, 1.0]).tolist() == [0x7E, 0xFE, 0x08, 0x01, 0x38]


def test_quantize_invariants():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(2, 3, 50, 64, generator=g) * 1.7).to(torch.bfloat16)
    codes, scale = fp8.quantize(x)
    x64 = x.double().numpy()
    amax = np.abs(x64).max(axis=(2, 3))
    assert np.allclose(scale, amax / 448.0, rtol=2 ** -23)
    # the amax element of each head maps to the largest code
    for b in range(2):
        for h in range(3):
            i = np.unravel_index(np.argmax(np.abs(x64[b, h])), x64[b, h].shape)
            assert codes[b, h][i] & 0x7F == 0x7E
    deq = fp8.dequantize(codes, scale)
    err = np.abs(deq - x64)
    assert np.all(err <= 2.0 ** -4 * np.abs(x64) + 2.0 ** -10 * scale[:, :, None, None] * 1.0001)
    # an all-zero head quantizes to zero codes with scale 1
    z = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    zc, zs = fp8.quantize(z)
    assert not zc.any() and zs[0, 0] == 1.0


def _rounded_o(qd, kd, vd, causal, sc, shift):
    """O with P = 2^(x - m_ref) rounded to e4m3, m_ref = row max - shift (log2 units)."""
    B, H, Nq, D = qd.shape
    Nkv = kd.shape[2]
    out = np.zeros_like(qd)
    legal = np.ones((Nq, Nkv), bool)
    if causal:
        legal = np.arange(Nkv)[None, :] <= np.arange(Nq)[:, None] + (Nkv - Nq)
    for b in range(B):
        for h in range(H):
            x = (sc * qd[b, h] @ kd[b, h].T) * np.log2(np.e)
            x = np.where(legal, x, -np.inf)
            m = x.max(axis=1, keepdims=True) - shift
            p = np.where(legal, np.exp2(x - m), 0.0).astype(np.float32)
            pr = fp8.e4m3_round(p)
            out[b, h] = (pr @ vd[b, h]) / p.astype(np.float64).sum(axis=1, keepdims=True)
    return out


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("amp", [0.5, 2.0])
def test_p_rounding_bound_holds_by_brute_force(causal, amp):
    oracle.build()
    g = torch.Generator().manual_seed(11)
    B, H, Nq, Nkv, D = 1, 2, 24, 300, 64
    q = (torch.randn(B, H, Nq, D, generator=g) * amp).to(torch.bfloat16)
    k = (torch.randn(B, H, Nkv, D, generator=g) * amp).to(torch.bfloat16)
    v = torch.randn(B, H, Nkv, D, generator=g).to(torch.bfloat16)
    o, lse, (qd, kd, vd) = fp8.attention_fwd_fp8(q, k, v, causal, 0.125)
    bound = fp8.p_rounding_bound(qd, kd, vd, causal, 0.125)
    worst = 0.0
    for shift in (0.0, 2.5, 8.0):
        orr = _rounded_o(qd, kd, vd, causal, 0.125, shift)
        assert np.all(np.abs(orr - o) <= bound + 1e-12)
        worst = max(worst, float((np.abs(orr - o) / np.maximum(bound, 1e-30)).max()))
    assert worst > 0.05  # the bound is not vacuous: the rounding reaches a fair share of it


def test_fp8_reference_is_the_plain_definition_of_dequantized_inputs():
    oracle.build()
    g = torch.Generator().manual_seed(5)
    q = torch.randn(1, 2, 7, 64, generator=g).to(torch.float16)
    k = torch.randn(1, 1, 9, 64, generator=g).to(torch.float16)
    v = torch.randn(1, 1, 9, 64, generator=g).to(torch.float16)
    o, lse, (qd, kd, vd) = fp8.attention_fwd_fp8(q, k, v, True, 0.2)
    # brute force with torch in fp64 on the dequantized values (GQA: repeat the kv head)
    qt, kt, vt = (torch.from_numpy(t) for t in (qd, kd, vd))
    kt, vt = kt.repeat_interleave(2, dim=1), vt.repeat_interleave(2, dim=1)
    s = 0.2 * qt @ kt.transpose(-1, -2)
    legal = torch.arange(9)[None, :] <= torch.arange(7)[:, None] + 2
    s = s.masked_fill(~legal, float("-inf"))
    ref_o = torch.softmax(s, dim=-1) @ vt
    ref_lse = torch.logsumexp(s, dim=-1)
    assert np.allclose(o, ref_o.numpy(), atol=1e-12)
    assert np.allclose(lse, ref_lse.numpy(), atol=1e-12)


def test_packed_fp8_single_sequence_is_the_dense_reference():
    # a packed batch of one sequence is one batch entry of the dense FP8 forward
    oracle.build()
    g = torch.Generator().manual_seed(11)
    q = torch.randn(1, 4, 13, 64, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 2, 21, 64, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 2, 21, 64, generator=g).to(torch.bfloat16)
    o, lse, (qd, kd, vd) = fp8.attention_fwd_fp8(q, k, v, True, 0.11)
    bound = fp8.p_rounding_bound(qd, kd, vd, True, 0.11)
    op, lp, bp = fp8.varlen_attention_fwd_fp8(q[0].transpose(0, 1), k[0].transpose(0, 1), v[0].transpose(0, 1),
                                              [0, 13], [0, 21], True, 0.11)
    assert np.array_equal(op, o[0].transpose(1, 0, 2))
    assert np.array_equal(lp, lse[0])
    assert np.array_equal(bp, bound[0].transpose(1, 0, 2))


def test_packed_fp8_scales_are_per_sequence():
    # scaling one sequence's inputs by a power of two changes nothing in the
    # other sequences (their scales are their own), and an empty-key sequence
    # gives O = 0 and LSE = -inf
    oracle.build()
    g = torch.Generator().manual_seed(12)
    cq, ck = [0, 9, 20, 26], [0, 11, 30, 30]
    q = torch.randn(26, 2, 64, generator=g).to(torch.bfloat16)
    k = torch.randn(30, 1, 64, generator=g).to(torch.bfloat16)
    v = torch.randn(30, 1, 64, generator=g).to(torch.bfloat16)
    o1, l1, _ = fp8.varlen_attention_fwd_fp8(q, k, v, cq, ck, False, 0.125)
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[9:20] *= 1024.0
    k2[11:30] *= 1024.0
    v2[11:30] *= 1024.0
    o2, l2, _ = fp8.varlen_attention_fwd_fp8(q2, k2, v2, cq, ck, False, 0.125)
    assert np.array_equal(o1[:9], o2[:9]) and np.array_equal(l1[:, :9], l2[:, :9])
    assert not np.allclose(o1[9:20], o2[9:20])
    assert np.all(o1[20:] == 0.0) and np.all(np.isneginf(l1[:, 20:]))
