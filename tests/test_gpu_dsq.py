"""GPU parity of the stored-tile backward (dense, D a multiple of 64 up to 1024,
either kernel family, causal or not):
the dK launch also writes dS^T to the workspace and dQ = scale dS K is one
GEMM; with room for P^T as well, the dK launch also writes P^T and
dV = P^T dO is one GEMM instead of a launch that recomputes S^T.

Every case runs the backward three times on the same inputs: with the small
workspace (dQ recomputes S and dP), with a middle one, and with room for dS
and P of every head. All three are checked against the fp64 oracle with the
usual gradient tolerance.
- With one kv head, the middle workspace holds dS for every head and stores
  dS only (dV recomputes): dV must be bit-identical to the small workspace's
  (the same kernel); dK too when non-causal (causal storing starts at an even
  query tile: an extra all-masked tile shifts the summation order), and dK
  must equal the big workspace's in the CTA-pair family (storing P does not
  change it there; the one-CTA family then forms dS^T from P rounded to fp16
  instead of fp32).
- With several kv heads, the middle workspace holds both tile sets of one kv
  group: the backward runs in chunks of one group (dK, then the dV and dQ
  GEMMs, per chunk), and every gradient must be bit-identical to the big
  workspace's (the same kernels on the same tiles).
"""
import math
import os

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


def pair_family(D):
    """Whether the backward kernels run as CTA pairs for this head dim."""
    forced = os.environ.get("FFPA_KERNEL")
    if forced in ("pair", "single"):
        return forced == "pair"
    return D % 128 == 0 and D <= 768


def tile_buffer_bytes(q, k):
    """Bytes of one stored-tile buffer: [B, Hq, Nkv, round_up(Nq, 8)] 16-bit values."""
    B, Hq, Nq, _ = q.shape
    Nkv = k.shape[2]
    return B * Hq * Nkv * ((Nq + 7) // 8 * 8) * 2


def run_both(B, Hq, Hkv, Nq, Nkv, D, dtype=torch.bfloat16, seed=0, causal=False):
    inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, dtype, seed=seed)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    scale = 1.0 / math.sqrt(D)
    o, lse = api.fwd(q, k, v, causal, scale)
    small_n = api.bwd_workspace_bytes(q, k)
    big_n = api.bwd_workspace_bytes(q, k, causal)
    one = tile_buffer_bytes(q, k)
    assert big_n >= small_n + 2 * one, "the stored-tile path applies to this problem"
    small = torch.empty(small_n, dtype=torch.uint8, device="cuda")
    ds_only = torch.empty(small_n + one, dtype=torch.uint8, device="cuda")
    big = torch.empty(big_n, dtype=torch.uint8, device="cuda")
    g_small = api.bwd(q, k, v, o, lse, do, causal, scale, workspace=small)
    mid = ds_only if Hkv == 1 else group_chunk_workspace(q, k, causal, 1)
    g_ds = api.bwd(q, k, v, o, lse, do, causal, scale, workspace=mid)
    g_big = api.bwd(q, k, v, o, lse, do, causal, scale, workspace=big)
    api.get_status()
    ref = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], causal, scale)
    for gs in (g_small, g_ds, g_big):
        for name, got, r in zip(("dQ", "dK", "dV"), gs, ref):
            check_grad(got, r, name)
    if Hkv == 1:  # dS stored, dV recomputed
        assert torch.equal(g_small[2], g_ds[2])
        if pair_family(D):
            assert torch.equal(g_ds[1], g_big[1])
        if not causal:
            assert torch.equal(g_small[1], g_ds[1])
    else:  # both tile sets in chunks of kv groups
        for name, a, b in zip(("dQ", "dK", "dV"), g_ds, g_big):
            assert torch.equal(a, b), f"{name}: chunked and one-chunk results differ"
    return inp, (q, k, v, do, o, lse, scale, big, ds_only), g_big, g_ds


@pytest.mark.parametrize("D", [256, 512])
@pytest.mark.parametrize("Nq,Nkv", [(256, 256), (301, 333), (1000, 129), (64, 700)])
def test_stored_ds_backward(D, Nq, Nkv):
    run_both(1, 2, 2, Nq, Nkv, D, seed=Nq + D)


@pytest.mark.parametrize("D", [128, 320, 384, 448, 576, 640, 768, 1024])
def test_stored_tile_backward_other_head_dims(D):
    # CTA pairs up to 768 (multiples of 128), one CTA per slab otherwise; GEMM
    # slabs that end 64 or 128 columns past a multiple of 256 end in an N = 128
    # MMA; D > 512 takes two slabs per row tile
    run_both(1, 2, 1, 300, 333, D, dtype=torch.float16, seed=D)


@pytest.mark.parametrize("D", [640, 1024])
def test_stored_tile_backward_other_head_dims_causal(D):
    run_both(1, 2, 2, 400, 300, D, seed=11, causal=True)


def test_stored_ds_backward_gqa_fp16():
    run_both(2, 8, 2, 300, 520, 512, dtype=torch.float16, seed=3)


def test_stage_bit_4_replays_the_gemm_on_the_stored_ds():
    # preprocess, dK (stores dS), then bit 4 alone: the same dQ as the full call
    # with room for dS only (dK computes S^T, as it does without bit 5)
    inp, (q, k, v, do, o, lse, scale, big, ds_only), _, (dq_full, _, _) = run_both(1, 4, 2, 512, 512, 512, seed=5)
    dq = torch.empty_like(q)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    for bit in (1, 8, 16):
        api.bwd(q, k, v, o, lse, do, False, scale, workspace=ds_only, dq=dq, dk=dk, dv=dv, stages=bit)
    api.get_status()
    assert torch.equal(dq, dq_full)


@pytest.mark.parametrize("causal", [False, True])
def test_stage_bit_5_splits_the_stored_p_launches(causal):
    # preprocess, dK storing P and dS, then the dV and dQ GEMMs: the same
    # gradients as the full call, launch by launch
    inp, (q, k, v, do, o, lse, scale, big, _), g_full, _ = run_both(1, 4, 2, 640, 384, 512, seed=7, causal=causal)
    dq = torch.empty_like(q)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    for bits in (1, 8 | 32, 2 | 32, 16):
        api.bwd(q, k, v, o, lse, do, causal, scale, workspace=big, dq=dq, dk=dk, dv=dv, stages=bits)
    api.get_status()
    for got, want in zip((dq, dk, dv), g_full):
        assert torch.equal(got, want)


def test_stage_bit_5_needs_the_p_buffer():
    q = torch.zeros(1, 2, 256, 512, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 2, 256, dtype=torch.float32, device="cuda")
    ds_only = torch.empty(api.bwd_workspace_bytes(q, q) + tile_buffer_bytes(q, q), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError, match="stage bit 5"):
        api.bwd(q, q, q, o, lse, o, False, 0.05, workspace=ds_only, stages=1 | 8 | 32)


@pytest.mark.parametrize("Nq,Nkv", [(300, 300), (256, 700), (700, 256), (100, 1000), (513, 769)])
def test_stored_ds_backward_causal(Nq, Nkv):
    # bottom-right causal: the dQ GEMM stops at each tile's last legal key, and
    # rows with no legal key (Nq > Nkv) get dQ = 0
    run_both(1, 4, 2, Nq, Nkv, 512, seed=Nq + 2 * Nkv, causal=True)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [512, 1024])
def test_stored_tile_varlen_backward(causal, D):
    # packed batches: every sequence's key rows start at cu_seqlens_k[b] + 256 b
    # in the tile buffers; empty sequences on either side, lengths that end
    # mid-tile, more queries than keys (causal rows with no legal key)
    lq = [5, 0, 130, 300, 64, 257]
    lk = [7, 3, 130, 200, 0, 513]
    inp = workloads.random_varlen(lq, lk, 4, 2, D, seed=71 + D)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    cq, ck = inp["cu_seqlens_q"].cuda(), inp["cu_seqlens_k"].cuda()
    scale = 1 / math.sqrt(D)
    o, lse = api.varlen_fwd(q, k, v, cq, ck, max(lq), max(lk), causal, scale)
    sizes = (0, len(lq), sum(lq), sum(lk), max(lq), max(lk), 4, 2, D)
    from head_dim_flash_gb300 import _ffi
    small_n = int(_ffi.ffpa_varlen_bwd_workspace_bytes(*sizes))
    big_n = int(_ffi.ffpa_varlen_bwd_workspace_bytes_ds(*sizes, int(causal)))
    rows = sum(lk) + 256 * len(lk)
    one = 4 * rows * ((max(lq) + 7) // 8 * 8) * 2
    assert big_n == small_n + (one + 255) // 256 * 256 + one
    ref = oracle.varlen_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                            causal, scale)
    got = {}
    for name, n in (("small", small_n), ("big", big_n)):
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        got[name] = api.varlen_bwd(q, k, v, o, lse, do, cq, ck, max(lq), max(lk), causal, scale, workspace=ws)
        api.get_status()
        for gname, g, r in zip(("dQ", "dK", "dV"), got[name], ref):
            check_grad(g, r, f"{name} {gname}")


def group_chunk_workspace(q, k, causal, groups):
    """A workspace with room for both tile sets of `groups` kv groups (the budget query's answer)."""
    B, Hq, Nq, _ = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    per_group = B * (Hq // Hkv) * Nkv * ((Nq + 7) // 8 * 8) * 2
    n = api.bwd_workspace_bytes(q, k, causal, budget=api.bwd_workspace_bytes(q, k) + 2 * groups * per_group + 512)
    assert api.bwd_workspace_bytes(q, k) < n < api.bwd_workspace_bytes(q, k, causal)
    return torch.empty(n, dtype=torch.uint8, device="cuda")


# Several chunks of kv groups (one or two groups per chunk, the last chunk
# evened out), dense: both kernel families, causal and not, GQA; against the
# fp64 oracle and bit for bit against the one-chunk path.
@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,D,causal,groups", [
    (1, 6, 3, 300, 333, 512, False, 1),
    (2, 8, 4, 257, 513, 512, True, 1),
    (1, 12, 6, 200, 300, 256, True, 2),
    (1, 4, 4, 130, 700, 320, False, 1),   # one-CTA family
    (1, 10, 5, 400, 300, 1024, True, 2),  # one-CTA family, two GEMM slabs, more queries than keys
    (2, 16, 4, 257, 300, 512, True, 1),   # GQA with 4 query heads per kv head, fp16 below
])
def test_stored_tiles_in_kv_group_chunks(B, Hq, Hkv, Nq, Nkv, D, causal, groups):
    dtype = torch.float16 if Hq // Hkv == 4 else torch.bfloat16
    inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, dtype, seed=Nq + D + Hq)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    scale = 1.0 / math.sqrt(D)
    o, lse = api.fwd(q, k, v, causal, scale)
    chunk_ws = group_chunk_workspace(q, k, causal, groups)
    full_ws = torch.empty(api.bwd_workspace_bytes(q, k, causal), dtype=torch.uint8, device="cuda")
    g_chunk = api.bwd(q, k, v, o, lse, do, causal, scale, workspace=chunk_ws)
    g_full = api.bwd(q, k, v, o, lse, do, causal, scale, workspace=full_ws)
    api.get_status()
    ref = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], causal, scale)
    for name, got, r, full in zip(("dQ", "dK", "dV"), g_chunk, ref, g_full):
        check_grad(got, r, name)
        assert torch.equal(got, full), f"{name}: chunked and one-chunk results differ"


@pytest.mark.parametrize("causal", [False, True])
def test_stored_tiles_in_kv_group_chunks_varlen(causal):
    from head_dim_flash_gb300 import _ffi

    lq = [5, 0, 130, 300, 64, 257]
    lk = [7, 3, 130, 200, 0, 513]
    Hq, Hkv, D = 6, 3, 512
    inp = workloads.random_varlen(lq, lk, Hq, Hkv, D, seed=91)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    cq, ck = inp["cu_seqlens_q"].cuda(), inp["cu_seqlens_k"].cuda()
    scale = 1 / math.sqrt(D)
    o, lse = api.varlen_fwd(q, k, v, cq, ck, max(lq), max(lk), causal, scale)
    sizes = (0, len(lq), sum(lq), sum(lk), max(lq), max(lk), Hq, Hkv, D)
    small_n = int(_ffi.ffpa_varlen_bwd_workspace_bytes(*sizes))
    big_n = int(_ffi.ffpa_varlen_bwd_workspace_bytes_ds(*sizes, int(causal)))
    per_group = (Hq // Hkv) * (sum(lk) + 256 * len(lk)) * ((max(lq) + 7) // 8 * 8) * 2
    chunk_n = api.varlen_workspace_bytes(q, k, cq, max(lq), max(lk), causal, budget=small_n + 2 * per_group + 512)
    assert small_n < chunk_n < big_n
    ref = oracle.varlen_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                            causal, scale)
    got = {}
    for name, n in (("chunks", chunk_n), ("one chunk", big_n)):
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        got[name] = api.varlen_bwd(q, k, v, o, lse, do, cq, ck, max(lq), max(lk), causal, scale, workspace=ws)
        api.get_status()
        for gname, g, r in zip(("dQ", "dK", "dV"), got[name], ref):
            check_grad(g, r, f"{name} {gname}")
    for gname, a, b in zip(("dQ", "dK", "dV"), got["chunks"], got["one chunk"]):
        assert torch.equal(a, b), f"{gname}: chunked and one-chunk results differ"


def test_default_workspace_is_fixed_by_the_budget():
    # the size bwd() allocates depends on the problem and the budget only: the
    # every-head tiles within the budget, a chunk of groups beyond it
    q = torch.zeros(1, 8, 1024, 512, dtype=torch.bfloat16, device="cuda")
    full = api.bwd_workspace_bytes(q, q, False)
    assert api.bwd_workspace(q, q, False).numel() == full
    per_group = 1024 * 1024 * 2
    n = api.bwd_workspace(q, q, False, budget=full - 1).numel()
    assert api.bwd_workspace_bytes(q, q) + 2 * 4 * per_group <= n < full  # 8 groups in 2 chunks of 4
    assert api.bwd_workspace(q, q, False, budget=1).numel() == api.bwd_workspace_bytes(q, q)


def test_varlen_and_other_head_dims_keep_the_recompute_path():
    for D in (96, 352):
        q = torch.zeros(1, 2, 64, D, dtype=torch.bfloat16, device="cuda")
        assert api.bwd_workspace_bytes(q, q, True) == api.bwd_workspace_bytes(q, q)
    for D in (128, 320, 512, 768, 1024):
        q5 = torch.zeros(1, 2, 64, D, dtype=torch.bfloat16, device="cuda")
        assert api.bwd_workspace_bytes(q5, q5, True) > api.bwd_workspace_bytes(q5, q5)


@pytest.mark.parametrize("family", ["single", "pair"])
def test_either_family_forced_stores_the_tiles(monkeypatch, family):
    # the dK kernels of both families store the tiles: forcing either one (the
    # one-CTA family at D = 512, CTA pairs at D = 576) keeps the parity
    monkeypatch.setenv("FFPA_KERNEL", family)
    if family == "pair":
        run_both(1, 2, 1, 200, 333, 576, dtype=torch.float16, seed=553, causal=True)
        return
    run_both(1, 4, 2, 150, 333, 512, dtype=torch.float16, seed=552, causal=True)
