"""The allocation-free routing entry point.

switch_moe_route_from_logits_noalloc serves callers that cannot allocate
device memory while they route (a server whose device memory all belongs to
a pool made at start-up, a runtime with a fixed memory budget): it takes no
workspace and keeps its scratch in a static device array.  This test calls
it through the C ABI and checks that it returns exactly what the workspace
entry point returns, on two calls in a row (the second call sees the first
call's leftovers in the shared array).  It sits in its own file, collected
last, and passes alone in a fresh process as well as after the other tests.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _raw_noalloc(lib, p, logits, o):
    return lib._lib.switch_moe_route_from_logits_noalloc(
        ctypes.byref(p), ctypes.c_void_p(logits.data_ptr()),
        *[ctypes.c_void_p(t.data_ptr()) for t in o],
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _outs(T, N):
    d = "cuda"
    return (torch.empty(T, dtype=torch.int32, device=d), torch.empty(T, device=d),
            torch.empty(T, dtype=torch.int32, device=d), torch.empty(T, dtype=torch.uint8, device=d),
            torch.empty(N, dtype=torch.int32, device=d), torch.empty(1, device=d))


@pytest.mark.parametrize("T,N,cf,mode", [(8192, 128, 1.25, 0), (16384, 64, 1.0, 1), (777, 5, 0.7, 1)])
def test_noalloc_matches_workspace_entry_point(lib, T, N, cf, mode):
    g = torch.Generator().manual_seed(T + N)
    for call in range(2):   # two calls in a row on different logits
        logits = (torch.randn(T, N, generator=g) * (1.0 + call)).cuda()
        ref = lib.switch_moe_route_from_logits(logits, cf, mode)
        p = lib.make_params(T, 8, 8, N, cf, mode, 1, lib.F32, 0)
        o = _outs(T, N)
        assert _raw_noalloc(lib, p, logits, o) == lib.SWITCH_MOE_OK
        assert lib.switch_moe_sync_status() == lib.SWITCH_MOE_OK
        # same kernels on the same logits: integers bit-exact, gate and aux
        # identical (within the routing tests' tolerances a fortiori)
        for got, want in zip(o, ref):
            assert torch.equal(got, want)


def test_noalloc_rejects_sizes_past_the_static_scratch(lib):
    logits = torch.zeros(16385, 4, device="cuda")
    p = lib.make_params(16385, 8, 8, 4, 1.0, 0, 1, lib.F32, 0)
    assert _raw_noalloc(lib, p, logits, _outs(16385, 4)) == lib.SWITCH_MOE_ERR_UNSUPPORTED
    logits = torch.zeros(64, 257, device="cuda")
    p = lib.make_params(64, 8, 8, 257, 1.0, 0, 1, lib.F32, 0)
    assert _raw_noalloc(lib, p, logits, _outs(64, 257)) == lib.SWITCH_MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,code", [
    (dict(expand=2), "UNSUPPORTED"), (dict(top_k=2), "UNSUPPORTED"),
    (dict(expert_choice=1), "UNSUPPORTED"), (dict(renormalize=1), "INVALID_ARG"),
])
def test_noalloc_takes_plain_top1_only(lib, kw, code):
    logits = torch.zeros(64, 8, device="cuda")
    p = lib.make_params(64, 8, 8, 8, 1.0, 0, 1, lib.F32, 0, **kw)
    assert _raw_noalloc(lib, p, logits, _outs(64, 8)) == getattr(lib, "SWITCH_MOE_ERR_" + code)
