"""ffpa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers run where no device allocation is possible (a fixed memory pool
planned ahead of time, a host framework that owns every buffer, a latency
path where cudaMalloc would synchronise the GPU), so they cannot hand
ffpa_bwd a workspace. ffpa_bwd_noalloc takes its scratch from an array built
into the library instead. This test calls it through the C ABI twice in a
row, on the same stream, and checks both results against ffpa_bwd with a
workspace, within the gradient tolerance the other GPU tests use. The second
call finds the first call's leftovers in the shared array and must not depend
on them. The file is named to be collected last, and it passes alone in a
fresh process as well as after the other tests.
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
    from head_dim_flash_gb300 import _ffi, api
    from head_dim_flash_gb300 import workloads
    from tests.gpu_utils import check_grad, to64

    stream = torch.cuda.current_stream().cuda_stream
    cases = [  # (B, Hq, Hkv, Nq, Nkv, D, causal, seed): the second call sees another shape's leftovers
        (1, 4, 2, 300, 333, 512, True, 3),
        (2, 2, 2, 129, 200, 320, False, 4),
    ]
    for B, Hq, Hkv, Nq, Nkv, D, causal, seed in cases:
        inp = workloads.random_dense(B, Hq, Hkv, Nq, Nkv, D, torch.bfloat16, seed=seed)
        t = {n: inp[n].cuda() for n in ("q", "k", "v", "dO")}
        scale = 1.0 / math.sqrt(D)
        t["o"], t["lse"] = api.fwd(t["q"], t["k"], t["v"], causal, scale)
        want = api.bwd(t["q"], t["k"], t["v"], t["o"], t["lse"], t["dO"], causal, scale)
        got = _grads_noalloc(_ffi, t, B, Hq, Hkv, Nq, Nkv, D, causal, scale, stream)
        for name, g, w in zip(("dQ", "dK", "dV"), got, want):
            check_grad(g, to64(w), name)

    # a problem past the built-in scratch is refused with an explanation, before any launch
    big = 1 << 20
    st = _ffi.ffpa_bwd_noalloc(_ffi.BF16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 1, 1, big, 8, 512, 0, 0.05, stream)
    assert st == _ffi.ERR_INVALID_VALUE
    assert "scratch" in _ffi.last_error()
