"""Error paths on a GPU.  Every bad argument here is rejected on the host
before anything is enqueued; the device-timeout path is exercised by the
diagnostic kernel whose bounded wait is bound to expire (no fault, no hang)."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _layer(T=256, d=64, F=128, N=4):
    x = torch.randn(T, d, device="cuda").bfloat16()
    W_g = torch.randn(N, d, device="cuda") * 0.1
    W1 = (torch.randn(N, F, d, device="cuda") * 0.1).bfloat16()
    W2 = (torch.randn(N, d, F, device="cuda") * 0.1).bfloat16()
    return x, W_g, W1, W2


def _raw_forward(lib, p, x_ptr, W_g, W1, W2, ws_ptr, ws_bytes, outs):
    return lib._lib.switch_moe_forward(
        ctypes.byref(p), ctypes.c_void_p(x_ptr), ctypes.c_void_p(W_g.data_ptr()), None,
        ctypes.c_void_p(W1.data_ptr()), ctypes.c_void_p(W2.data_ptr()), None, None,
        *[ctypes.c_void_p(o.data_ptr()) for o in outs], ctypes.c_void_p(ws_ptr),
        ctypes.c_size_t(ws_bytes), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _outs(T, d, N):
    return [torch.empty((T, d), device="cuda"), torch.empty(T, dtype=torch.int32, device="cuda"),
            torch.empty(T, device="cuda"), torch.empty(T, dtype=torch.int32, device="cuda"),
            torch.empty(T, dtype=torch.uint8, device="cuda"),
            torch.empty(N, dtype=torch.int32, device="cuda"), torch.empty(1, device="cuda")]


def test_workspace_too_small(lib):
    x, W_g, W1, W2 = _layer()
    p = lib.make_params(256, 64, 128, 4, 1.0)
    need = lib.switch_moe_workspace_bytes(p)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    rc = _raw_forward(lib, p, x.data_ptr(), W_g, W1, W2, ws.data_ptr(), need - 1,
                      _outs(256, 64, 4))
    assert rc == lib.SWITCH_MOE_ERR_WORKSPACE_TOO_SMALL


def test_misaligned_pointers(lib):
    x, W_g, W1, W2 = _layer()
    p = lib.make_params(256, 64, 128, 4, 1.0)
    need = lib.switch_moe_workspace_bytes(p)
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    outs = _outs(256, 64, 4)
    # x two bytes past a 16-byte boundary
    xb = torch.empty(256 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    rc = _raw_forward(lib, p, xb.data_ptr() + 2, W_g, W1, W2, ws.data_ptr(), need, outs)
    assert rc == lib.SWITCH_MOE_ERR_ALIGNMENT
    # workspace not 256-byte aligned
    rc = _raw_forward(lib, p, x.data_ptr(), W_g, W1, W2, ws.data_ptr() + 128, need, outs)
    assert rc == lib.SWITCH_MOE_ERR_ALIGNMENT


def test_null_and_bad_params(lib):
    x, W_g, W1, W2 = _layer()
    p = lib.make_params(256, 64, 128, 4, 1.0)
    need = lib.switch_moe_workspace_bytes(p)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    outs = _outs(256, 64, 4)
    assert _raw_forward(lib, p, 0, W_g, W1, W2, ws.data_ptr(), need, outs) == \
        lib.SWITCH_MOE_ERR_INVALID_ARG
    bad = lib.make_params(256, 64, 128, 4, -1.0)
    assert _raw_forward(lib, bad, x.data_ptr(), W_g, W1, W2, ws.data_ptr(), need, outs) == \
        lib.SWITCH_MOE_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        lib.switch_moe_forward(x, W_g, W1.transpose(1, 2), W2, 1.0)


def test_device_timeout_is_reported_and_cleared(lib):
    assert lib.switch_moe_sync_status() == lib.SWITCH_MOE_OK
    lib.switch_moe_selftest_wait_timeout(20_000_000)      # 20 ms bounded wait, bound to expire
    assert lib.switch_moe_sync_status() == lib.SWITCH_MOE_ERR_DEVICE_TIMEOUT
    assert lib.switch_moe_sync_status() == lib.SWITCH_MOE_OK   # cleared by the read
    # the context is still healthy: a forward runs afterwards
    x, W_g, W1, W2 = _layer()
    o = lib.switch_moe_forward(x, W_g, W1, W2, 1.0)
    assert lib.switch_moe_sync_status() == lib.SWITCH_MOE_OK
    assert torch.isfinite(o.y).all()
