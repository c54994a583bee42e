"""ffpa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers run where no device allocation is possible (a fixed memory pool
planned ahead of time, a host framework that owns every buffer, a latency
path where cudaMalloc would synchronise the GPU), so they cannot hand
ffpa_bwd a workspace. ffpa_bwd_noalloc takes its scratch from an array built
into the library instead. This test calls it through the C ABI several times
in a row, on the same stream, and checks every result against ffpa_bwd with a
workspace (which takes the stored-tile kernels here, while the no-alloc call
always recomputes), and one case against the fp64 oracle, within the
gradient tolerance the other GPU tests use. Each call after the first finds
the previous call's leftovers in the shared array (a non-causal problem
before a causal one, a larger problem before a smaller one) and must not
depend on them. The file is named to be collected last, and it passes alone in
a fresh process as well as after the other tests.
"""
import math

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_dim_flash_gb300 import build

    build.build()


def _grads_noalloc(ffi, t, B, Hq, Hkv, Nq, Nkv, D, causal, scale, stream):
    dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
    st = ffi.ffpa_bwd_noalloc(ffi.BF16, t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), t["o"].data_ptr(),
                              t["lse"].data_ptr(), t["dO"].data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                              B, Hq, Hkv, Nq, Nkv, D, int(causal), scale, stream)
    ffi.raise_for(st, "ffpa_bwd_noalloc")
    ffi.raise_for(ffi.ffpa_get_status(stream), "device status")
    return dq, dk, dv


def test_noalloc_backward_matches_workspace_backward_twice_in_a_row():
    import oracle
    from head_dim_flash_gb300 import _ffi, api
    from head_dim_flash_gb300 import workloads
    from tests.gpu_utils import check_grad, to64

    oracle.build()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [  # (B, Hq, Hkv, Nq, Nkv, D, causal, seed, against the oracle too)
        (2, 2, 2, 129, 200, 320, False, 4, False),   # leaves the array non-zero
        (1, 4, 2, 300, 333, 512, True, 3, True),     # causal after non-causal
        (1, 8, 8, 1024, 1024, 512, True, 5, False),  # larger: its dS^T would not fit the array
        (1, 2, 1, 77, 90, 256, False, 6, False),     # smaller after larger
    ]
    for B, Hq, Hkv, Nq, Nkv, D, causal, seed, vs_oracle in cases:
        inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, torch.bfloat16, seed=seed)
        t = {n: inp[n].cuda() for n in ("q", "k", "v", "dO")}
        scale = 1.0 / math.sqrt(D)
        t["o"], t["lse"] = api.fwd(t["q"], t["k"], t["v"], causal, scale)
        want = api.bwd(t["q"], t["k"], t["v"], t["o"], t["lse"], t["dO"], causal, scale)
        got = _grads_noalloc(_ffi, t, B, Hq, Hkv, Nq, Nkv, D, causal, scale, stream)
        for name, g, w in zip(("dQ", "dK", "dV"), got, want):
            check_grad(g, to64(w), name)
        if vs_oracle:
            ref = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], causal, scale)
            for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
                check_grad(g, r, name + " (oracle)")

    # a problem past the built-in scratch is refused with an explanation, before any launch
    big = 1 << 20
    st = _ffi.ffpa_bwd_noalloc(_ffi.BF16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 1, 1, big, 8, 512, 0, 0.05, stream)
    assert st == _ffi.ERR_INVALID_VALUE
    assert "scratch" in _ffi.last_error()
