"""Host-side checks of the C ABI that need no GPU.

The library must load and export every symbol include/ffpa.h declares, and
every invalid call must be rejected with the documented status before any
device work (so these calls are safe without a GPU). The product path must
fail loudly when the library is missing.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import torch

    from head_dim_flash_gb300 import _ffi, build

    # these calls pass fake device addresses that every rejected call leaves
    # untouched; where a GPU is visible, a validation slip would launch on them,
    # so they run only on a machine without one
    if torch.cuda.is_available():
        pytest.skip("host-only ABI checks (fake device pointers) run where no GPU is visible")
    build.build()
    return _ffi.load()


def header_symbols():
    txt = open(os.path.join(ROOT, "include", "ffpa.h")).read()
    return sorted(set(re.findall(r"FFPA_API\s+[\w\s\*]+?\b(ffpa_\w+)\s*\(", txt)))


def test_header_declares_the_documented_entry_points():
    syms = header_symbols()
    for name in ("ffpa_fwd", "ffpa_bwd", "ffpa_varlen_fwd", "ffpa_varlen_bwd", "ffpa_bwd_workspace_bytes",
                 "ffpa_varlen_bwd_workspace_bytes", "ffpa_get_status", "ffpa_last_error"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    from head_dim_flash_gb300 import _ffi

    syms = header_symbols()
    assert set(syms) == set(_ffi.EXPORTS)
    for name in syms:
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_missing_library_fails_loudly(tmp_path):
    from head_dim_flash_gb300 import _ffi

    with pytest.raises(RuntimeError, match="missing"):
        _ffi.load(str(tmp_path / "nope.so"))


FAKE = 0x10000  # 16-byte aligned fake device address; never dereferenced by rejected calls


def fwd(lib, dt=0, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, Hq=2, Hkv=1, Nq=8, Nkv=8, D=512, causal=0,
        scale=0.05):
    return lib.ffpa_fwd(dt, q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, D, causal, scale, None)


@pytest.mark.parametrize("kw,status", [
    (dict(dt=5), 2),                 # dtype outside bf16/fp16
    (dict(D=100), 2),                # D not a multiple of 64
    (dict(D=1088), 2),               # D above 1024
    (dict(D=32), 2),                 # D below 64
    (dict(Hq=3, Hkv=2), 1),          # Hq not a multiple of Hkv
    (dict(Hkv=0), 1),
    (dict(scale=float("nan")), 1),
    (dict(scale=float("inf")), 1),
    (dict(Nq=-1), 1),
    (dict(q=0), 1),                  # NULL with a non-empty problem
    (dict(lse=0), 1),
    (dict(k=FAKE + 2), 1),           # misaligned
    (dict(B=1, Hq=1 << 20, Hkv=1 << 20, Nq=1 << 22), 2),  # more work units than 65535^2 clusters
    (dict(B=1 << 19, Hq=1 << 12, Hkv=1 << 12), 2),       # B*Hq beyond int
])
def test_invalid_forward_calls_are_rejected(lib, kw, status):
    assert fwd(lib, **kw) == status
    assert lib.ffpa_last_error()  # a message explains the rejection


def test_head_dims_multiple_of_32_pass_the_dim_check(lib):
    # D = 96, 160: accepted by the head-dim check (a later check, here the NaN
    # scale, rejects the call before any device work); D = 100, 80: not
    for D in (96, 160, 992):
        assert fwd(lib, D=D, scale=float("nan")) == 1
    for D in (100, 80, 1056):
        assert fwd(lib, D=D, scale=float("nan")) == 2


def test_empty_problem_is_ok_without_launch(lib):
    assert fwd(lib, B=0, q=0, k=0, v=0, o=0, lse=0) == 0
    assert fwd(lib, Nq=0, q=0, o=0, lse=0, k=0, v=0) == 0


def test_workspace_size_and_checks(lib):
    n = lib.ffpa_bwd_workspace_bytes(0, 1, 32, 32, 8192, 8192, 512)
    assert n >= 2 * 32 * 8192 * 4 and n % 256 == 0
    args = [0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE]
    # workspace too small
    assert lib.ffpa_bwd(*args, FAKE, 16, 1, 32, 32, 8192, 8192, 512, 0, 0.05, None) == 1
    # workspace misaligned
    assert lib.ffpa_bwd(*args, FAKE + 16, n, 1, 32, 32, 8192, 8192, 512, 0, 0.05, None) == 1
    assert lib.ffpa_varlen_bwd_workspace_bytes(0, 2, 100, 100, 60, 60, 4, 2, 512) >= 2 * 4 * 100 * 4


def test_stored_tile_workspace_and_stage_bits(lib):
    # dense D = 512: row statistics, then dS^T, then P^T at the next 256-byte boundary
    B, Hq, Hkv, Nq, Nkv, D = 1, 4, 2, 300, 200, 512
    small = lib.ffpa_bwd_workspace_bytes(0, B, Hq, Hkv, Nq, Nkv, D)
    tile = B * Hq * Nkv * ((Nq + 7) // 8 * 8) * 2
    big = lib.ffpa_bwd_workspace_bytes_ds(0, B, Hq, Hkv, Nq, Nkv, D, 1)
    assert big == small + (tile + 255) // 256 * 256 + tile
    # head dims outside the path (not whole 64-column chunks) keep the small workspace
    assert lib.ffpa_bwd_workspace_bytes_ds(0, B, Hq, Hkv, Nq, Nkv, 352, 0) == lib.ffpa_bwd_workspace_bytes(
        0, B, Hq, Hkv, Nq, Nkv, 352)
    ptrs = [FAKE] * 9  # q, k, v, o, lse, dO, dq, dk, dv

    def stages(ws_bytes, bits):
        return lib.ffpa_bwd_stages(0, *ptrs, FAKE, ws_bytes, B, Hq, Hkv, Nq, Nkv, D, 0, 0.05, bits, None)

    # packed batches: Hq x (total_k + 256 batch) x round_up(max_q, 8) per buffer
    vsmall = lib.ffpa_varlen_bwd_workspace_bytes(0, 3, 700, 500, 300, 250, Hq, Hkv, D)
    vtile = Hq * (500 + 256 * 3) * 304 * 2
    assert lib.ffpa_varlen_bwd_workspace_bytes_ds(0, 3, 700, 500, 300, 250, Hq, Hkv, D, 1) == (
        vsmall + (vtile + 255) // 256 * 256 + vtile)
    assert lib.ffpa_varlen_bwd_workspace_bytes_ds(0, 3, 700, 500, 300, 250, Hq, Hkv, 352, 1) == (
        lib.ffpa_varlen_bwd_workspace_bytes(0, 3, 700, 500, 300, 250, Hq, Hkv, 352))
    assert stages(big, 64) == 1 and "bits 0..5" in lib.ffpa_last_error().decode()
    assert stages(small, 16) == 1 and "stage bit 4" in lib.ffpa_last_error().decode()
    assert stages(small + tile, 1 | 8 | 32) == 1 and "stage bit 5" in lib.ffpa_last_error().decode()
    assert stages(small, 2 | 32) == 1 and "stage bit 5" in lib.ffpa_last_error().decode()


def test_varlen_requires_both_cu_seqlens(lib):
    st = lib.ffpa_varlen_fwd(0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 10, 10, 5, 5, 4, 2, 512, 0, 0.05, None)
    assert st == 1
    assert "one-sided" in lib.ffpa_last_error().decode()


def test_python_api_maps_status_to_exceptions():
    from head_dim_flash_gb300 import _ffi

    with pytest.raises(NotImplementedError):
        _ffi.raise_for(_ffi.ERR_NOT_SUPPORTED, "x")
    with pytest.raises(ValueError):
        _ffi.raise_for(_ffi.ERR_INVALID_VALUE, "x")
    with pytest.raises(TimeoutError):
        _ffi.raise_for(_ffi.ERR_TIMEOUT, "x")
    with pytest.raises(RuntimeError):
        _ffi.raise_for(_ffi.ERR_CUDA, "x")


def test_python_api_rejects_unsupported_dtype_before_the_library():
    import torch

    from head_dim_flash_gb300 import api

    with pytest.raises(NotImplementedError):
        api._dt(torch.zeros(1, dtype=torch.float32))


def _view(ptr=FAKE, sb=2 * 8 * 512, sh=8 * 512, sn=512):
    from head_dim_flash_gb300 import _ffi

    return _ffi.View(ptr, sb, sh, sn)


@pytest.mark.parametrize("which,bad", [
    ("q", dict(sn=100)),             # stride not a multiple of 8 elements
    ("q", dict(sh=0)),               # zero stride along Hq = 2 heads
    ("o", dict(ptr=FAKE + 8)),       # misaligned data
    ("v", dict(sb=-8)),              # negative stride
    ("k", dict(sn=1 << 39)),         # beyond the tensor-map stride limit
    ("o", dict(ptr=0)),              # NULL with a non-empty problem
])
def test_invalid_strided_views_are_rejected(lib, which, bad):
    views = {name: _view() for name in ("q", "k", "v", "o")}
    views[which] = _view(**bad)
    st = lib.ffpa_fwd_strided(0, views["q"], views["k"], views["v"], views["o"], FAKE, 1, 2, 1, 8, 8, 512, 0, 0.05,
                              None)
    assert st == 1
    assert which.encode() in lib.ffpa_last_error()


def test_strided_backward_checks_every_view(lib):
    good = _view()
    args = [good] * 4 + [FAKE] + [good, good, good, _view(sn=12)]  # dv stride not a multiple of 8
    n = lib.ffpa_bwd_workspace_bytes(0, 1, 2, 1, 8, 8, 512)
    assert lib.ffpa_bwd_strided(0, *args, FAKE, n, 1, 2, 1, 8, 8, 512, 0, 0.05, None) == 1
    assert b"dv" in lib.ffpa_last_error()


def test_python_views_are_zero_copy_for_common_layouts():
    import torch

    from head_dim_flash_gb300 import api

    B, N, H, D = 2, 5, 3, 64
    bnhd = torch.zeros(B, N, H, D, dtype=torch.bfloat16)
    assert api._viewable(torch.zeros(B, H, N, D, dtype=torch.bfloat16))
    assert api._viewable(bnhd.transpose(1, 2))                       # [B, N, H, D] storage
    fused = torch.zeros(B, N, 3, H, D, dtype=torch.bfloat16)
    assert api._viewable(fused[:, :, 1].transpose(1, 2))             # K slice of a fused QKV buffer
    assert not api._viewable(torch.zeros(B, H, D, N, dtype=torch.bfloat16).transpose(2, 3))  # head dim strided
    assert not api._viewable(torch.zeros(B, H, N, D + 4, dtype=torch.bfloat16)[..., :D])      # row stride 68


def _decode(lib, Hq=8, Hkv=1, Nq=1, Nkv=4096, D=512, ws=FAKE, ws_bytes=None, q=None, lse=FAKE, scale=0.05):
    vq = q if q is not None else _view(sb=Hq * Nq * D, sh=Nq * D, sn=D)
    vk = _view(sb=Hkv * Nkv * D, sh=Nkv * D, sn=D)
    vo = _view(sb=Hq * Nq * D, sh=Nq * D, sn=D)
    if ws_bytes is None:
        ws_bytes = lib.ffpa_decode_workspace_bytes(0, 1, Hq, Hkv, Nq, Nkv, D)
    return lib.ffpa_decode_fwd(0, vq, vk, vk, vo, lse, ws, ws_bytes, 1, Hq, Hkv, Nq, Nkv, D, 0, scale, None)


def test_decode_workspace_covers_every_split_partial():
    from head_dim_flash_gb300 import _ffi

    lib = _ffi.load()
    for Hq, Hkv, Nq, Nkv, D in ((8, 1, 1, 4096, 512), (32, 4, 2, 100, 320), (4, 4, 16, 70000, 1024)):
        n = lib.ffpa_decode_workspace_bytes(0, 2, Hq, Hkv, Nq, Nkv, D)
        rows = 2 * Hq * Nq
        assert n >= rows * (D + 1) * 4          # at least one split
        assert n % (rows * (D + 1) * 4) == 0    # a whole number of splits
        assert n // (rows * (D + 1) * 4) <= 64
    assert lib.ffpa_decode_workspace_bytes(0, 1, 3, 2, 1, 8, 512) == 0  # Hq not a multiple of Hkv


@pytest.mark.parametrize("kw,status,msg", [
    (dict(Hq=1 << 17, Hkv=1, Nq=1 << 20, Nkv=64), 2, "grid"),  # 2^33 row blocks > 65535^2
    (dict(D=352), 2, "multiple of 64"),              # D % 64 == 32: tile kernels only
    (dict(ws_bytes=16), 1, "workspace"),             # workspace too small
    (dict(ws=FAKE + 16), 1, "aligned"),              # workspace not 256-byte aligned
    (dict(ws=0), 1, "aligned"),
    (dict(lse=0), 1, "lse"),
    (dict(scale=float("nan")), 1, "scale"),
])
def test_invalid_decode_calls_are_rejected(lib, kw, status, msg):
    assert _decode(lib, **kw) == status
    assert msg in lib.ffpa_last_error().decode()


def test_decode_checks_views(lib):
    assert _decode(lib, q=_view(sn=12)) == 1  # row stride not a multiple of 8 elements
    assert b"q" in lib.ffpa_last_error()


def test_decode_supported_predicate():
    import torch

    from head_dim_flash_gb300 import api

    q = torch.zeros(2, 8, 2, 512)
    assert api.decode_supported(q, torch.zeros(2, 1, 9, 512))        # 16 rows per kv head: one row block
    assert api.decode_supported(torch.zeros(2, 8, 3, 512), torch.zeros(2, 1, 9, 512))  # 24 rows: two blocks
    assert not api.decode_supported(q, torch.zeros(2, 0, 9, 512))    # no kv heads
    assert not api.decode_supported(q, torch.zeros(2, 3, 9, 512))    # Hq not a multiple of Hkv
    assert not api.decode_supported(torch.zeros(2, 8, 1, 352), torch.zeros(2, 1, 9, 352))  # D % 64 != 0
    big = torch.zeros(1, 1, 1, 64).expand(1, 64, 16400, 64)          # 64 x 1025 row blocks (shape only)
    assert api.decode_supported(big, torch.zeros(1, 64, 9, 64))      # beyond one grid dimension: fine
    huge = torch.zeros(1, 1, 1, 64).expand(1, 1 << 17, 1 << 20, 64)  # 2^33 row blocks (shape only)
    assert not api.decode_supported(huge, torch.zeros(1, 1, 9, 64))  # beyond the 65535^2 units of a grid


def _fp8(lib, fn="fwd", D=512, Nq=8, Nkv=8, ws=FAKE, ws_bytes=None, Hq=2, Hkv=1, lse=FAKE):
    vq = _view(sb=Hq * Nq * D, sh=Nq * D, sn=D)
    vk = _view(sb=Hkv * Nkv * D, sh=Nkv * D, sn=D)
    if ws_bytes is None:
        ws_bytes = lib.ffpa_fp8_workspace_bytes(1, Hq, Hkv, Nq, Nkv, D)
    if fn == "fwd":
        return lib.ffpa_fwd_fp8(0, vq, vk, vk, vq, lse, ws, ws_bytes, 1, Hq, Hkv, Nq, Nkv, D, 0, 0.05, None)
    return lib.ffpa_fp8_quantize(0, vq, vk, vk, ws, ws_bytes, 1, Hq, Hkv, Nq, Nkv, D, None)


@pytest.mark.parametrize("fn", ["fwd", "quantize"])
@pytest.mark.parametrize("kw,status,msg", [
    (dict(D=48), 2, "multiple of 32"),     # below the FP8 range 64..1024
    (dict(D=1056), 2, "multiple of 32"),   # above it
    (dict(Nkv=0), 2, "Nkv"),
    (dict(ws_bytes=1024), 1, "workspace too small"),
    (dict(ws=FAKE + 64), 1, "aligned"),
])
def test_invalid_fp8_calls_are_rejected(lib, fn, kw, status, msg):
    assert _fp8(lib, fn, **kw) == status
    assert msg in lib.ffpa_last_error().decode()


def test_fp8_forward_checks_lse(lib):
    assert _fp8(lib, "fwd", lse=0) == 1
    assert b"lse" in lib.ffpa_last_error()


def test_fp8_workspace_layout():
    from head_dim_flash_gb300 import _ffi

    for D, Dp in ((512, 512), (320, 384), (96, 128), (1024, 1024)):  # code rows padded to 128
        B, Hq, Hkv, Nq, Nkv = 2, 8, 2, 300, 777
        off = _ffi.ffpa_fp8_workspace_layout(B, Hq, Hkv, Nq, Nkv, D)
        q8, k8, v8t, sq, sk, sv, ldv, total = off
        assert ldv == 784  # Nkv rounded up to 16
        assert all(o % 256 == 0 for o in (q8, k8, v8t, sq, sk, sv, total))
        assert k8 >= q8 + B * Hq * Nq * Dp and v8t >= k8 + B * Hkv * Nkv * Dp and sq >= v8t + B * Hkv * Dp * ldv
        assert sk >= sq + 4 * B * Hq and sv >= sk + 4 * B * Hkv and total > sv
        assert _ffi.ffpa_fp8_workspace_bytes(B, Hq, Hkv, Nq, Nkv, D) == total
    assert _ffi.ffpa_fp8_workspace_bytes(1, 2, 1, 8, 8, 48) == 0  # outside the head-dim range


def test_fp8_prequantized_entry_validates_before_any_launch(lib):
    n = lib.ffpa_fp8_workspace_bytes(1, 2, 1, 8, 8, 512)
    vo = _view(sb=2 * 8 * 512, sh=8 * 512, sn=512)
    # workspace too small, misaligned, unsupported head dim, missing lse
    assert lib.ffpa_fwd_fp8_quantized(0, vo, FAKE, FAKE, 64, 1, 2, 1, 8, 8, 512, 0, 0.05, None) == 1
    assert lib.ffpa_fwd_fp8_quantized(0, vo, FAKE, FAKE + 32, n, 1, 2, 1, 8, 8, 512, 0, 0.05, None) == 1
    assert lib.ffpa_fwd_fp8_quantized(0, _view(sb=2 * 8 * 1056, sh=8 * 1056, sn=1056), FAKE, FAKE, n,
                                      1, 2, 1, 8, 8, 1056, 0, 0.05, None) == 2
    assert lib.ffpa_fwd_fp8_quantized(0, vo, 0, FAKE, n, 1, 2, 1, 8, 8, 512, 0, 0.05, None) == 1
    assert b"lse" in lib.ffpa_last_error()


def test_backward_workspace_budget_plan(lib):
    # the stored-tile workspace within a budget: every head's tiles when they
    # fit, else both tile sets of an evened-out chunk of kv groups, else the
    # row statistics alone; host arithmetic only (no device)
    B, Hq, Hkv, Nq, Nkv, D = 2, 8, 4, 300, 333, 512
    small = lib.ffpa_bwd_workspace_bytes(0, B, Hq, Hkv, Nq, Nkv, D)
    full = lib.ffpa_bwd_workspace_bytes_ds(0, B, Hq, Hkv, Nq, Nkv, D, 1)
    group = B * (Hq // Hkv) * Nkv * 304 * 2  # one kv group's query heads, queries rounded up to 8

    def plan(budget):
        return lib.ffpa_bwd_workspace_bytes_budget(0, B, Hq, Hkv, Nq, Nkv, D, 1, budget)

    def a256(x):
        return (x + 255) // 256 * 256

    assert plan(1 << 40) == full
    assert plan(full) == full
    assert plan(full - 1) == small + a256(2 * group) + 2 * group       # 3 groups fit: 2 chunks of 2
    assert plan(small + 2 * group + 512) == small + a256(group) + group  # 1 group per chunk
    assert plan(small + 2 * group - 1) == small                        # not even one group
    assert plan(0) == small
    # head dims the stored-tile path does not take keep the small workspace
    assert lib.ffpa_bwd_workspace_bytes_budget(0, B, Hq, Hkv, Nq, Nkv, 352, 1, 1 << 40) == small
    # packed batches: one group's rows are every sequence's keys plus a 256-row pad each
    vsmall = lib.ffpa_varlen_bwd_workspace_bytes(0, 3, 600, 700, 300, 400, 4, 2, 512)
    vgroup = 2 * (700 + 3 * 256) * 304 * 2
    assert lib.ffpa_varlen_bwd_workspace_bytes_budget(0, 3, 600, 700, 300, 400, 4, 2, 512, 0,
                                                      vsmall + 2 * vgroup + 512) == vsmall + a256(vgroup) + vgroup


def test_packed_fp8_validates_before_any_launch(lib):
    n = lib.ffpa_varlen_fp8_workspace_bytes(2, 30, 40, 20, 25, 4, 2, 512)
    assert n > 0

    def call(cu_k=FAKE, total_k=40, ws=FAKE, ws_bytes=n, D=512, lse=FAKE):
        return lib.ffpa_varlen_fwd_fp8(0, FAKE, FAKE, FAKE, FAKE, lse, FAKE, cu_k, 2, 30, total_k, 20, 25, 4, 2, D,
                                       1, 0.05, ws, ws_bytes, None)

    assert call(cu_k=None) == 1 and "one-sided" in lib.ffpa_last_error().decode()
    assert call(ws_bytes=n - 1) == 1 and "too small" in lib.ffpa_last_error().decode()
    assert call(ws=FAKE + 32) == 1 and "256-byte" in lib.ffpa_last_error().decode()
    assert call(total_k=0, ws_bytes=lib.ffpa_varlen_fp8_workspace_bytes(2, 30, 0, 20, 25, 4, 2, 512)) == 2
    assert call(D=48) == 2
    assert call(lse=0) == 1
    # sizes: V^T columns for 16-aligned sequence starts, per-(sequence, head) scales
    assert lib.ffpa_varlen_fp8_workspace_bytes(2, 30, 40, 20, 25, 4, 2, 48) == 0
    assert lib.ffpa_varlen_fp8_workspace_bytes(3, 30, 40, 20, 25, 4, 2, 512) > n
