"""Pins for the fp64 oracle, checked against things other than itself.

Exact softmax attention has a plain definition (FFPA docs, "Backends
Overview" page, "Automatic SDPA fallback": the SDPA-aligned result; "CuTe-DSL
Backend" page, "Hard constraints": bottom-right causal, zero-stride GQA, empty
rows give O=0, LSE=-inf and zero gradients; "Varlen (packed THD) API": packed
layout and LSE [H, T]). These tests pin the oracle to:
  * a hand-derived worked example (tests/golden/hand_example.json),
  * torch library routines (softmax / logsumexp / autograd) in fp64 on tiny
    shapes with the mask built explicitly,
  * closed forms (uniform scores, one legal key, empty rows, key shift),
  * invariants (convexity, gradient sums), finite differences,
  * structural identities (GQA == MHA with repeated K/V, varlen == per-
    sequence dense calls),
and show that plausible mistakes planted in a copy of the oracle fail them.
"""
import json
import math
import os
import shutil

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


# ----------------------------------------------------------------------------
# independent brute force on torch library routines (fp64)
# ----------------------------------------------------------------------------
def bottom_right_mask(nq, nk, causal):
    i = torch.arange(nq).view(-1, 1)
    j = torch.arange(nk).view(1, -1)
    if not causal:
        return torch.ones(nq, nk, dtype=torch.bool)
    return j <= i + (nk - nq)


def brute_attention(q, k, v, causal, scale):
    """q [B,Hq,Nq,D], k,v [B,Hkv,Nkv,D] fp64 tensors -> (O, LSE)."""
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    g = Hq // Hkv
    kk = k.repeat_interleave(g, dim=1)
    vv = v.repeat_interleave(g, dim=1)
    s = scale * torch.einsum("bhid,bhjd->bhij", q, kk)
    mask = bottom_right_mask(Nq, Nk, causal)
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    empty = ~mask.any(dim=-1)
    p = torch.softmax(s, dim=-1)
    p = torch.where(empty.view(1, 1, -1, 1), torch.zeros_like(p), p)
    o = torch.einsum("bhij,bhjd->bhid", p, vv)
    return o, lse


def t64(x):
    return torch.as_tensor(np.asarray(x), dtype=torch.float64)


def rnd(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64)


SHAPES = [
    # B, Hq, Hkv, Nq, Nkv, D
    (1, 1, 1, 8, 8, 16),
    (2, 4, 2, 5, 9, 8),
    (1, 4, 1, 9, 5, 32),  # Nq > Nkv: causal rows 0..3 are empty
    (2, 2, 2, 16, 16, 64),
    (1, 3, 3, 1, 7, 16),
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_torch_bruteforce(shape, causal):
    B, Hq, Hkv, Nq, Nk, D = shape
    q, k, v = rnd((B, Hq, Nq, D), 1), rnd((B, Hkv, Nk, D), 2), rnd((B, Hkv, Nk, D), 3)
    scale = 0.7 / math.sqrt(D)
    o, lse = oracle.attention_fwd(q, k, v, causal, scale)
    o_ref, lse_ref = brute_attention(q, k, v, causal, scale)
    np.testing.assert_allclose(o, o_ref.numpy(), rtol=1e-12, atol=1e-12)
    fin = np.isfinite(lse_ref.numpy())
    np.testing.assert_array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], lse_ref.numpy()[fin], rtol=1e-12, atol=1e-12)
    assert np.all(lse[~fin] == -np.inf)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd(shape, causal):
    B, Hq, Hkv, Nq, Nk, D = shape
    q, k, v = rnd((B, Hq, Nq, D), 4), rnd((B, Hkv, Nk, D), 5), rnd((B, Hkv, Nk, D), 6)
    do = rnd((B, Hq, Nq, D), 7)
    scale = 1.3 / math.sqrt(D)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, scale)
    qr, kr, vr = (x.clone().requires_grad_(True) for x in (q, k, v))
    o_ref, _ = brute_attention(qr, kr, vr, causal, scale)
    (o_ref * do).sum().backward()
    np.testing.assert_allclose(dq, qr.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, kr.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, vr.grad.numpy(), rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------------------
# hand-derived worked example
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("mode", ["noncausal", "causal"])
def test_hand_worked_example(mode):
    ex = json.load(open(os.path.join(HERE, "golden", "hand_example.json")))
    q = np.array(ex["q"])[None, None]
    k = np.array(ex["k"])[None, None]
    v = np.array(ex["v"])[None, None]
    do = np.array(ex["dO"])[None, None]
    causal = mode == "causal"
    o, lse = oracle.attention_fwd(q, k, v, causal, ex["scale"])
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, ex["scale"])
    want = ex[mode]
    np.testing.assert_allclose(o[0, 0], want["O"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], want["LSE"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(dq[0, 0], want["dQ"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dk[0, 0], want["dK"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dv[0, 0], want["dV"], rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(6, 6), (4, 9), (9, 4)])
def test_uniform_scores_give_mean_of_legal_values(causal, nq, nk):
    D = 16
    q = np.zeros((1, 2, nq, D))
    k = rnd((1, 2, nk, D), 11).numpy()
    v = rnd((1, 2, nk, D), 12).numpy()
    o, lse = oracle.attention_fwd(q, k, v, causal, 0.3)
    for i in range(nq):
        n_legal = nk if not causal else max(0, min(nk, i + (nk - nq) + 1))
        if n_legal == 0:
            assert np.all(o[:, :, i] == 0) and np.all(lse[:, :, i] == -np.inf)
            continue
        np.testing.assert_allclose(o[:, :, i], v[:, :, :n_legal].mean(axis=2), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[:, :, i], math.log(n_legal), rtol=1e-14, atol=1e-14)


def test_single_legal_key_returns_that_value_row():
    D, N = 32, 7
    q, k, v = rnd((1, 1, N, D), 13), rnd((1, 1, N, D), 14), rnd((1, 1, N, D), 15)
    scale = 1 / math.sqrt(D)
    o, lse = oracle.attention_fwd(q, k, v, True, scale)
    np.testing.assert_array_equal(o[0, 0, 0], v[0, 0, 0].numpy())
    np.testing.assert_allclose(lse[0, 0, 0], scale * float(q[0, 0, 0] @ k[0, 0, 0]), rtol=1e-14)


def test_empty_rows_zero_output_and_exactly_zero_gradients():
    # causal with Nq=8 > Nkv=4: bottom-right alignment leaves rows 0..3 without a legal key
    B, H, Nq, Nk, D = 1, 2, 8, 4, 16
    q, k, v = rnd((B, H, Nq, D), 16), rnd((B, H, Nk, D), 17), rnd((B, H, Nk, D), 18)
    do = rnd((B, H, Nq, D), 19)
    o, lse = oracle.attention_fwd(q, k, v, True, 0.25)
    assert np.all(o[:, :, :4] == 0.0)
    assert np.all(lse[:, :, :4] == -np.inf)
    assert np.all(np.isfinite(lse[:, :, 4:]))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, True, 0.25)
    assert np.all(dq[:, :, :4] == 0.0)
    # dO on empty rows must not reach dK/dV at all
    do2 = do.clone()
    do2[:, :, :4] = 1e6
    _, dk2, dv2 = oracle.attention_bwd(q, k, v, do2, True, 0.25)
    np.testing.assert_array_equal(dk, dk2)
    np.testing.assert_array_equal(dv, dv2)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_moves_lse_only(causal):
    B, H, Nq, Nk, D = 1, 2, 6, 10, 8
    q, k, v = rnd((B, H, Nq, D), 20), rnd((B, H, Nk, D), 21), rnd((B, H, Nk, D), 22)
    c = rnd((D,), 23)
    scale = 0.5
    o1, lse1 = oracle.attention_fwd(q, k, v, causal, scale)
    o2, lse2 = oracle.attention_fwd(q, k + c, v, causal, scale)
    np.testing.assert_allclose(o2, o1, rtol=1e-11, atol=1e-12)
    shift = scale * torch.einsum("bhid,d->bhi", q, c).numpy()
    np.testing.assert_allclose(lse2 - lse1, shift, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_output_is_a_convex_combination(causal):
    B, H, Nq, Nk, D = 2, 2, 9, 13, 8
    q, k, v = rnd((B, H, Nq, D), 24) * 3, rnd((B, H, Nk, D), 25), rnd((B, H, Nk, D), 26)
    o, _ = oracle.attention_fwd(q, k, v, causal, 1.0)
    vn = v.numpy()
    for i in range(Nq):
        n_legal = Nk if not causal else min(Nk, i + (Nk - Nq) + 1)
        lo = vn[:, :, :n_legal].min(axis=2)
        hi = vn[:, :, :n_legal].max(axis=2)
        assert np.all(o[:, :, i] >= lo - 1e-12) and np.all(o[:, :, i] <= hi + 1e-12)


# ----------------------------------------------------------------------------
# gradients: finite differences and invariants
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_central_finite_differences(causal):
    B, H, N, D = 1, 1, 8, 32
    q, k, v = rnd((B, H, N, D), 27).numpy(), rnd((B, H, N, D), 28).numpy(), rnd((B, H, N, D), 29).numpy()
    do = rnd((B, H, N, D), 30).numpy()
    scale = 1 / math.sqrt(D)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, scale)

    def loss(qq, kk, vv):
        o, _ = oracle.attention_fwd(qq, kk, vv, causal, scale)
        return float((o * do).sum())

    h = 1e-6
    rng = np.random.default_rng(0)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(24):
            idx = tuple(int(rng.integers(0, s)) for s in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd = (loss(**{"qq": args_p["q"], "kk": args_p["k"], "vv": args_p["v"]})
                  - loss(**{"qq": args_m["q"], "kk": args_m["k"], "vv": args_m["v"]})) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-7 * max(1.0, abs(g[idx])) + 2e-9, (name, idx, fd, g[idx])


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sum_invariants(causal):
    # sum_j dS_ij = 0 for every row  =>  sum_j dK_j = 0 per kv head;
    # sum_j P_ij = 1 on non-empty rows => sum_j dV_j = sum over the group of non-empty dO_i
    B, Hq, Hkv, Nq, Nk, D = 2, 4, 2, 9, 6, 16
    q, k, v = rnd((B, Hq, Nq, D), 31), rnd((B, Hkv, Nk, D), 32), rnd((B, Hkv, Nk, D), 33)
    do = rnd((B, Hq, Nq, D), 34)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, 0.4)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    mask = bottom_right_mask(Nq, Nk, causal).any(dim=-1).numpy()
    want = do.numpy()[:, :, mask].sum(axis=2).reshape(B, Hkv, Hq // Hkv, D).sum(axis=2)
    np.testing.assert_allclose(dv.sum(axis=2), want, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------
# structural identities: GQA and varlen
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_with_repeated_kv(causal):
    B, Hq, Hkv, Nq, Nk, D = 1, 6, 2, 7, 11, 8
    q, k, v = rnd((B, Hq, Nq, D), 35), rnd((B, Hkv, Nk, D), 36), rnd((B, Hkv, Nk, D), 37)
    do = rnd((B, Hq, Nq, D), 38)
    g = Hq // Hkv
    kr, vr = k.repeat_interleave(g, 1), v.repeat_interleave(g, 1)
    o1, l1 = oracle.attention_fwd(q, k, v, causal, 0.3)
    o2, l2 = oracle.attention_fwd(q, kr, vr, causal, 0.3)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-13, atol=1e-14)
    dq1, dk1, dv1 = oracle.attention_bwd(q, k, v, do, causal, 0.3)
    dq2, dk2, dv2 = oracle.attention_bwd(q, kr, vr, do, causal, 0.3)
    np.testing.assert_allclose(dq1, dq2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dk1, dk2.reshape(B, Hkv, g, Nk, D).sum(2), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv1, dv2.reshape(B, Hkv, g, Nk, D).sum(2), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_per_sequence_dense(causal):
    lq = [5, 0, 9, 3]
    lk = [7, 4, 9, 0]  # a query-less sequence and a key-less sequence (rows empty)
    Hq, Hkv, D = 4, 2, 8
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    q, k, v = rnd((sum(lq), Hq, D), 39), rnd((sum(lk), Hkv, D), 40), rnd((sum(lk), Hkv, D), 41)
    do = rnd((sum(lq), Hq, D), 42)
    o, lse = oracle.varlen_fwd(q, k, v, cq, ck, causal, 0.35)
    dq, dk, dv = oracle.varlen_bwd(q, k, v, do, cq, ck, causal, 0.35)
    assert lse.shape == (Hq, sum(lq))
    for b in range(len(lq)):
        qs, ks = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
        if lq[b] == 0:
            if lk[b]:
                assert np.all(dk[ks] == 0) and np.all(dv[ks] == 0)
            continue
        qb = q[qs].permute(1, 0, 2)[None]
        kb, vb = k[ks].permute(1, 0, 2)[None], v[ks].permute(1, 0, 2)[None]
        dob = do[qs].permute(1, 0, 2)[None]
        ob, lb = oracle.attention_fwd(qb, kb, vb, causal, 0.35)
        np.testing.assert_allclose(o[qs], ob[0].transpose(1, 0, 2), rtol=1e-13, atol=1e-14)
        np.testing.assert_array_equal(lse[:, qs], lb[0])
        if lk[b] == 0:
            assert np.all(o[qs] == 0) and np.all(lse[:, qs] == -np.inf) and np.all(dq[qs] == 0)
            continue
        dqb, dkb, dvb = oracle.attention_bwd(qb, kb, vb, dob, causal, 0.35)
        np.testing.assert_allclose(dq[qs], dqb[0].transpose(1, 0, 2), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dk[ks], dkb[0].transpose(1, 0, 2), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dv[ks], dvb[0].transpose(1, 0, 2), rtol=1e-12, atol=1e-13)


def test_row_sample_matches_full_forward():
    N, D = 40, 16
    q, k, v = rnd((N, D), 43), rnd((N + 3, D), 44), rnd((N + 3, D), 45)
    rows = [0, 5, 39, 17]
    for causal in (False, True):
        o, lse = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], causal, 0.2)
        os_, ls = oracle.attention_fwd_rows(q, k, v, rows, causal, 0.2)
        np.testing.assert_array_equal(os_, o[0, 0, rows])
        np.testing.assert_array_equal(ls, lse[0, 0, rows])


# ----------------------------------------------------------------------------
# pin strength: plant plausible mistakes in a copy of the oracle, on the CPU
# ----------------------------------------------------------------------------
MUTATIONS = {
    # causal alignment top-left instead of bottom-right
    "top_left_causal": ("return j <= i + (lk - lq);", "return j <= i;"),
    # dropped scale in dK
    "dk_without_scale": ("dkj[d] += scale * ds * qi[d];", "dkj[d] += ds * qi[d];"),
    # GQA mapping interleaved instead of grouped
    "gqa_modulo": ("const long hk = h / g;", "const long hk = h % L->Hkv;"),
    # sign error in dS
    "ds_sign": ("const double ds = p * (dp - hv->delta[i]);\n        for (long d = 0; d < D; ++d) dqi",
                "const double ds = p * (hv->delta[i] - dp);\n        for (long d = 0; d < D; ++d) dqi"),
    # LSE without the max shift
    "lse_no_max": ("const double lse = m + log(l);", "const double lse = log(l);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(oracle._SRC).read()
    assert old in src, name
    mutated = tmp_path / "mutated.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = oracle.load_library(oracle.build(force=True, src=str(mutated), out=str(tmp_path / "libmut.so")))
    caught = []
    oracle.use_library(lib)
    try:
        for test, kwargs in (
            (test_forward_matches_torch_bruteforce, {"shape": (2, 4, 2, 5, 9, 8), "causal": True}),
            (test_backward_matches_torch_autograd, {"shape": (2, 4, 2, 5, 9, 8), "causal": True}),
            (test_hand_worked_example, {"mode": "causal"}),
        ):
            try:
                test(**kwargs)
            except AssertionError:
                caught.append(test.__name__)
    finally:
        oracle.use_library(None)
    assert caught, f"mutation {name} escaped every pin"
