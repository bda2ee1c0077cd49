"""Python binding of libswitchmoe.so: the forward pass of a Switch-style
top-1 Mixture-of-Experts FFN layer on one B300 (sm_103a).

This module only marshals arguments: it checks tensor shapes, dtypes and
devices, allocates outputs and workspace through PyTorch, and calls the C ABI
declared in include/switch_moe.h with raw device pointers and the current
CUDA stream.  Every step of the layer runs in the library's CUDA kernels;
there is no other implementation to fall back to, and importing this module
fails if the library has not been built.

Functions carry the C ABI's names:

    switch_moe_forward(x, W_g, W1, W2, capacity_factor, ...) -> ForwardOut
    switch_moe_route_from_logits(logits, capacity_factor, ...) -> RouteOut
    switch_moe_forward_expert_choice(x, W_g, W1, W2, capacity_factor, ...) -> ExpertChoiceOut
    switch_moe_route_expert_choice(logits, capacity_factor) -> ExpertChoiceOut (y None)
    switch_moe_backward(x, W_g, W1, W2, capacity_factor, fwd, dy, ...) -> BackwardOut
    switch_moe_router_logits(x, W_g, b_g=None) -> logits [T, N] fp32
    switch_moe_forward_hostio(x_host, W_g, W1, W2, ...) -> ForwardOut (host tensors)
    switch_moe_capacity(T, N, cf) -> int
    switch_moe_workspace_bytes(params) / switch_moe_hostio_workspace_bytes(params)
    switch_moe_sync_status() -> int, switch_moe_strerror(code) -> str
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libswitchmoe.so")

SWITCH_MOE_OK = 0
SWITCH_MOE_ERR_INVALID_ARG = -1
SWITCH_MOE_ERR_ALIGNMENT = -2
SWITCH_MOE_ERR_WORKSPACE_TOO_SMALL = -3
SWITCH_MOE_ERR_UNSUPPORTED = -4
SWITCH_MOE_ERR_CUDA = -5
SWITCH_MOE_ERR_DEVICE_TIMEOUT = -6
SWITCH_MOE_ERR_NO_DEVICE = -7
TOKEN_ORDER = 0
GATE_PRIORITY = 1
F32 = 0
BF16 = 1

EXPORTED = (
    "switch_moe_capacity", "switch_moe_workspace_bytes", "switch_moe_forward",
    "switch_moe_route_from_logits", "switch_moe_router_logits",
    "switch_moe_hostio_workspace_bytes", "switch_moe_forward_hostio",
    "switch_moe_sync_status", "switch_moe_strerror", "switch_moe_version",
    "switch_moe_selftest_wait_timeout", "switch_moe_set_phase_events",
    "switch_moe_route_from_logits_noalloc", "switch_moe_forward_expert_choice",
    "switch_moe_route_expert_choice", "switch_moe_backward_workspace_bytes",
    "switch_moe_backward",
)
NUM_PHASE_EVENTS = 8
PHASES = ("router", "scan_aux", "slots_dispatch", "shared_gemms", "expert_gemm1",
          "expert_gemm2", "combine")


class Params(ctypes.Structure):
    """Mirror of switch_moe_params."""
    _fields_ = [
        ("T", ctypes.c_int64), ("d_model", ctypes.c_int64), ("d_ff", ctypes.c_int64),
        ("N", ctypes.c_int64), ("capacity_factor", ctypes.c_double),
        ("priority_mode", ctypes.c_int32), ("gate_multiply", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("has_shared", ctypes.c_int32),
        ("expand", ctypes.c_int32), ("top_k", ctypes.c_int32),
        ("renormalize", ctypes.c_int32), ("expert_choice", ctypes.c_int32),
    ]


class SwitchMoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {strerror(code)} ({code})")
        self.code = code


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m switch_top_expert_router_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, V, I64, I32 = ctypes.POINTER(Params), ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    SZ = ctypes.POINTER(ctypes.c_size_t)
    lib.switch_moe_capacity.argtypes = [I64, I64, ctypes.c_double]
    lib.switch_moe_capacity.restype = I64
    for name in ("switch_moe_workspace_bytes", "switch_moe_hostio_workspace_bytes"):
        getattr(lib, name).argtypes = [P, SZ]
        getattr(lib, name).restype = I32
    fwd = [P, V, V, V, V, V, V, V, V, V, V, V, V, V, V, V, ctypes.c_size_t, V]
    lib.switch_moe_forward.argtypes = fwd
    lib.switch_moe_forward.restype = I32
    # p, 7 inputs, 6 outputs, workspace, its size, stream
    lib.switch_moe_forward_expert_choice.argtypes = [P] + [V] * 14 + [ctypes.c_size_t, V]
    lib.switch_moe_forward_expert_choice.restype = I32
    lib.switch_moe_route_expert_choice.argtypes = [P, V, V, V, V, V, V, V, ctypes.c_size_t, V]
    lib.switch_moe_route_expert_choice.restype = I32
    lib.switch_moe_backward_workspace_bytes.argtypes = [P, SZ]
    lib.switch_moe_backward_workspace_bytes.restype = I32
    # p, 7 inputs, 4 routing outputs, dy, aux_coef, 7 gradients, workspace, size, stream
    lib.switch_moe_backward.argtypes = ([P] + [V] * 12 + [ctypes.c_float] + [V] * 8
                                        + [ctypes.c_size_t, V])
    lib.switch_moe_backward.restype = I32
    lib.switch_moe_forward_hostio.argtypes = fwd
    lib.switch_moe_forward_hostio.restype = I32
    lib.switch_moe_route_from_logits.argtypes = [P, V, V, V, V, V, V, V, V, ctypes.c_size_t, V]
    lib.switch_moe_route_from_logits.restype = I32
    lib.switch_moe_route_from_logits_noalloc.argtypes = [P, V, V, V, V, V, V, V, V]
    lib.switch_moe_route_from_logits_noalloc.restype = I32
    lib.switch_moe_router_logits.argtypes = [P, V, V, V, V, V, ctypes.c_size_t, V]
    lib.switch_moe_router_logits.restype = I32
    lib.switch_moe_sync_status.argtypes = [V]
    lib.switch_moe_sync_status.restype = I32
    lib.switch_moe_strerror.argtypes = [I32]
    lib.switch_moe_strerror.restype = ctypes.c_char_p
    lib.switch_moe_selftest_wait_timeout.argtypes = [ctypes.c_uint64, V]
    lib.switch_moe_selftest_wait_timeout.restype = I32
    lib.switch_moe_set_phase_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), I32]
    lib.switch_moe_set_phase_events.restype = I32
    lib.switch_moe_version.argtypes = []
    lib.switch_moe_version.restype = I32
    return lib


class _Lazy:
    """Loads the library on first use, so that building it never needs a
    previous build; any call fails loudly when the .so is missing."""
    _h = None

    def __getattr__(self, name):
        if _Lazy._h is None:
            _Lazy._h = _load()
        return getattr(_Lazy._h, name)


_lib = _Lazy()


def load_library() -> ctypes.CDLL:
    """Load (once) and return the ctypes handle of libswitchmoe.so."""
    _lib.switch_moe_version  # noqa: B018  (forces the load)
    return _Lazy._h


class ForwardOut(NamedTuple):
    y: torch.Tensor              # [T, d_model] fp32
    expert_id: torch.Tensor      # [T] int32
    gate: torch.Tensor           # [T] fp32
    slot: torch.Tensor           # [T] int32 (-1 = dropped)
    drop_mask: torch.Tensor      # [T] uint8
    expert_counts: torch.Tensor  # [N] int32
    aux_loss: torch.Tensor       # [1] fp32


class ExpertChoiceOut(NamedTuple):
    y: Optional[torch.Tensor]    # [T, d_model] fp32 (None from the routing-only call)
    chosen_token: torch.Tensor   # [N, C] int32: each expert's tokens, best first; -1 past T
    chosen_gate: torch.Tensor    # [N, C] fp32: their scores
    experts_per_token: torch.Tensor  # [T] int32
    expert_counts: torch.Tensor  # [N] int32: the router's top-1 counts
    aux_loss: torch.Tensor       # [1] fp32: L_aux of the router's top-1 choice


class RouteOut(NamedTuple):
    expert_id: torch.Tensor
    gate: torch.Tensor
    slot: torch.Tensor
    drop_mask: torch.Tensor
    expert_counts: torch.Tensor
    aux_loss: torch.Tensor


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(code: int, where: str):
    if code != SWITCH_MOE_OK:
        raise SwitchMoEError(code, where)


def strerror(code: int) -> str:
    return _lib.switch_moe_strerror(int(code)).decode()


switch_moe_strerror = strerror


def switch_moe_version() -> int:
    return int(_lib.switch_moe_version())


def switch_moe_capacity(T: int, N: int, capacity_factor: float) -> int:
    c = int(_lib.switch_moe_capacity(int(T), int(N), float(capacity_factor)))
    if c < 1:
        raise SwitchMoEError(c, "switch_moe_capacity")
    return c


def make_params(T, d_model, d_ff, N, capacity_factor, priority_mode=TOKEN_ORDER,
                gate_multiply=1, dtype=BF16, has_shared=0, expand=1, top_k=1,
                renormalize=0, expert_choice=0) -> Params:
    return Params(int(T), int(d_model), int(d_ff), int(N), float(capacity_factor),
                  int(priority_mode), int(gate_multiply), int(dtype), int(has_shared),
                  int(expand), int(top_k), int(renormalize), int(expert_choice))


def _token_shape(T: int, top_k: int) -> tuple:
    """Shape of the per-token routing outputs: [T], or [T, 2] for top-2."""
    return (T, 2) if top_k == 2 else (T,)


def _check_out(out, T: int, d: int, N: int, top_k: int, names) -> None:
    """Output tensors the caller passed must have the sizes the library writes."""
    want = [T * d] + [T * (2 if top_k == 2 else 1)] * (len(names) - 3) + [N, 1]
    for t, n, name in zip(out, want, names):
        if t.numel() != n or not t.is_contiguous():
            raise ValueError(f"out.{name} must be contiguous with {n} elements")


def switch_moe_workspace_bytes(p: Params) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.switch_moe_workspace_bytes(ctypes.byref(p), ctypes.byref(n)),
           "switch_moe_workspace_bytes")
    return int(n.value)


def switch_moe_hostio_workspace_bytes(p: Params) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.switch_moe_hostio_workspace_bytes(ctypes.byref(p), ctypes.byref(n)),
           "switch_moe_hostio_workspace_bytes")
    return int(n.value)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"x must be bf16 or fp32, got {t.dtype}")


def _contig(t, name, dtype=None, device=None):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    return t


def workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _layer_args(x, W_g, W1, W2, b_g, W1s, W2s, device):
    dt = x.dtype
    _contig(W_g, "W_g", torch.float32, device)
    _contig(W1, "W1", dt, device)
    _contig(W2, "W2", dt, device)
    _contig(b_g, "b_g", torch.float32, device)
    _contig(W1s, "W1s", dt, device)
    _contig(W2s, "W2s", dt, device)
    T, d = x.shape
    N, F, d1 = W1.shape
    if W_g.shape != (N, d) or d1 != d or W2.shape != (N, d, F):
        raise ValueError(f"shape mismatch: x {tuple(x.shape)}, W_g {tuple(W_g.shape)}, "
                         f"W1 {tuple(W1.shape)}, W2 {tuple(W2.shape)}")
    if b_g is not None and b_g.shape != (N,):
        raise ValueError("b_g must be [N]")
    if (W1s is None) != (W2s is None):
        raise ValueError("W1s and W2s go together")
    if W1s is not None and (W1s.shape != (F, d) or W2s.shape != (d, F)):
        raise ValueError("shared expert must be W1s [d_ff, d_model], W2s [d_model, d_ff]")
    return T, d, F, N


def switch_moe_forward(x: torch.Tensor, W_g: torch.Tensor, W1: torch.Tensor, W2: torch.Tensor,
                       capacity_factor: float, priority_mode: int = TOKEN_ORDER,
                       gate_multiply: int = 1, b_g: Optional[torch.Tensor] = None,
                       W1s: Optional[torch.Tensor] = None, W2s: Optional[torch.Tensor] = None,
                       ws: Optional[torch.Tensor] = None, out: Optional[ForwardOut] = None,
                       stream=None, expand: int = 1, top_k: int = 1,
                       renormalize: int = 0) -> ForwardOut:
    """The whole layer; see switch_moe_forward in include/switch_moe.h
    (expand: Expanded Drop candidates, 1 = off; top_k: 1 or 2 experts per
    token, renormalize: top-2 gates over the chosen pair)."""
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor (use switch_moe_forward_hostio for host data)")
    dev = x.device
    _contig(x, "x", None, dev)
    T, d, F, N = _layer_args(x, W_g, W1, W2, b_g, W1s, W2s, dev)
    p = make_params(T, d, F, N, capacity_factor, priority_mode, gate_multiply, _dtype_code(x),
                    int(W1s is not None), expand, top_k, renormalize)
    need = switch_moe_workspace_bytes(p)
    if ws is None:
        ws = workspace(need, dev)
    ts = _token_shape(T, top_k)
    if out is None:
        out = ForwardOut(torch.empty((T, d), dtype=torch.float32, device=dev),
                         torch.empty(ts, dtype=torch.int32, device=dev),
                         torch.empty(ts, dtype=torch.float32, device=dev),
                         torch.empty(ts, dtype=torch.int32, device=dev),
                         torch.empty(ts, dtype=torch.uint8, device=dev),
                         torch.empty(N, dtype=torch.int32, device=dev),
                         torch.empty(1, dtype=torch.float32, device=dev))
    _check_out(out, T, d, N, top_k, ForwardOut._fields)
    with torch.cuda.device(dev):
        rc = _lib.switch_moe_forward(
            ctypes.byref(p), _ptr(x), _ptr(W_g), _ptr(b_g), _ptr(W1), _ptr(W2), _ptr(W1s),
            _ptr(W2s), _ptr(out.y), _ptr(out.expert_id), _ptr(out.gate), _ptr(out.slot),
            _ptr(out.drop_mask), _ptr(out.expert_counts), _ptr(out.aux_loss), _ptr(ws),
            ctypes.c_size_t(ws.numel()), _stream(stream))
    _check(rc, "switch_moe_forward")
    return out


def switch_moe_forward_hostio(x_host: torch.Tensor, W_g: torch.Tensor, W1: torch.Tensor,
                              W2: torch.Tensor, capacity_factor: float,
                              priority_mode: int = TOKEN_ORDER, gate_multiply: int = 1,
                              b_g: Optional[torch.Tensor] = None,
                              W1s: Optional[torch.Tensor] = None,
                              W2s: Optional[torch.Tensor] = None,
                              ws: Optional[torch.Tensor] = None,
                              out: Optional[ForwardOut] = None, stream=None,
                              expand: int = 1, top_k: int = 1,
                              renormalize: int = 0) -> ForwardOut:
    """Host input and output tensors (pin them for asynchronous copies);
    device weights.  Outputs are valid after the stream is synchronised."""
    if x_host.is_cuda:
        raise ValueError("x_host must be a host tensor")
    dev = W1.device
    _contig(x_host, "x_host")
    T, d, F, N = _layer_args(x_host, W_g, W1, W2, b_g, W1s, W2s, dev)
    p = make_params(T, d, F, N, capacity_factor, priority_mode, gate_multiply,
                    _dtype_code(x_host), int(W1s is not None), expand, top_k, renormalize)
    need = switch_moe_hostio_workspace_bytes(p)
    if ws is None:
        ws = workspace(need, dev)
    ts = _token_shape(T, top_k)
    if out is None:
        pin = torch.cuda.is_available()
        out = ForwardOut(torch.empty((T, d), dtype=torch.float32, pin_memory=pin),
                         torch.empty(ts, dtype=torch.int32, pin_memory=pin),
                         torch.empty(ts, dtype=torch.float32, pin_memory=pin),
                         torch.empty(ts, dtype=torch.int32, pin_memory=pin),
                         torch.empty(ts, dtype=torch.uint8, pin_memory=pin),
                         torch.empty(N, dtype=torch.int32, pin_memory=pin),
                         torch.empty(1, dtype=torch.float32, pin_memory=pin))
    _check_out(out, T, d, N, top_k, ForwardOut._fields)
    with torch.cuda.device(dev):
        rc = _lib.switch_moe_forward_hostio(
            ctypes.byref(p), _ptr(x_host), _ptr(W_g), _ptr(b_g), _ptr(W1), _ptr(W2),
            _ptr(W1s), _ptr(W2s), _ptr(out.y), _ptr(out.expert_id), _ptr(out.gate),
            _ptr(out.slot), _ptr(out.drop_mask), _ptr(out.expert_counts), _ptr(out.aux_loss),
            _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream))
    _check(rc, "switch_moe_forward_hostio")
    return out


def switch_moe_route_from_logits(logits: torch.Tensor, capacity_factor: float,
                                 priority_mode: int = TOKEN_ORDER,
                                 ws: Optional[torch.Tensor] = None,
                                 stream=None, expand: int = 1, top_k: int = 1,
                                 renormalize: int = 0) -> RouteOut:
    """Routing on given fp32 logits [T, N] (expand: Expanded Drop candidates;
    top_k: 1 or 2 experts per token; renormalize: top-2 gates over the pair)."""
    dev = logits.device
    _contig(logits, "logits", torch.float32)
    T, N = logits.shape
    p = make_params(T, 8, 8, N, capacity_factor, priority_mode, 1, F32, 0, expand, top_k,
                    renormalize)
    need = switch_moe_workspace_bytes(p)
    if ws is None:
        ws = workspace(need, dev)
    ts = _token_shape(T, top_k)
    o = RouteOut(torch.empty(ts, dtype=torch.int32, device=dev),
                 torch.empty(ts, dtype=torch.float32, device=dev),
                 torch.empty(ts, dtype=torch.int32, device=dev),
                 torch.empty(ts, dtype=torch.uint8, device=dev),
                 torch.empty(N, dtype=torch.int32, device=dev),
                 torch.empty(1, dtype=torch.float32, device=dev))
    with torch.cuda.device(dev):
        rc = _lib.switch_moe_route_from_logits(
            ctypes.byref(p), _ptr(logits), _ptr(o.expert_id), _ptr(o.gate), _ptr(o.slot),
            _ptr(o.drop_mask), _ptr(o.expert_counts), _ptr(o.aux_loss), _ptr(ws),
            ctypes.c_size_t(ws.numel()), _stream(stream))
    _check(rc, "switch_moe_route_from_logits")
    return o


def switch_moe_route_from_logits_noalloc(logits: torch.Tensor, capacity_factor: float,
                                         priority_mode: int = TOKEN_ORDER,
                                         out: Optional[RouteOut] = None,
                                         stream=None) -> RouteOut:
    """Routing on given fp32 logits without a workspace, for callers that
    cannot allocate device memory at routing time (the library keeps the
    scratch in a static device array).  At most 16384 tokens and 256
    experts.  Pass preallocated ``out`` tensors to allocate nothing here
    either."""
    dev = logits.device
    _contig(logits, "logits", torch.float32)
    T, N = logits.shape
    p = make_params(T, 8, 8, N, capacity_factor, priority_mode, 1, F32, 0)
    if out is None:
        out = RouteOut(torch.empty(T, dtype=torch.int32, device=dev),
                       torch.empty(T, dtype=torch.float32, device=dev),
                       torch.empty(T, dtype=torch.int32, device=dev),
                       torch.empty(T, dtype=torch.uint8, device=dev),
                       torch.empty(N, dtype=torch.int32, device=dev),
                       torch.empty(1, dtype=torch.float32, device=dev))
    with torch.cuda.device(dev):
        rc = _lib.switch_moe_route_from_logits_noalloc(
            ctypes.byref(p), _ptr(logits), _ptr(out.expert_id), _ptr(out.gate), _ptr(out.slot),
            _ptr(out.drop_mask), _ptr(out.expert_counts), _ptr(out.aux_loss), _stream(stream))
    _check(rc, "switch_moe_route_from_logits_noalloc")
    return out


def _ec_outputs(T: int, d: Optional[int], N: int, C: int, dev) -> ExpertChoiceOut:
    return ExpertChoiceOut(
        None if d is None else torch.empty((T, d), dtype=torch.float32, device=dev),
        torch.empty((N, C), dtype=torch.int32, device=dev),
        torch.empty((N, C), dtype=torch.float32, device=dev),
        torch.empty(T, dtype=torch.int32, device=dev),
        torch.empty(N, dtype=torch.int32, device=dev),
        torch.empty(1, dtype=torch.float32, device=dev))


def switch_moe_forward_expert_choice(x: torch.Tensor, W_g: torch.Tensor, W1: torch.Tensor,
                                     W2: torch.Tensor, capacity_factor: float,
                                     gate_multiply: int = 1, b_g: Optional[torch.Tensor] = None,
                                     W1s: Optional[torch.Tensor] = None,
                                     W2s: Optional[torch.Tensor] = None,
                                     ws: Optional[torch.Tensor] = None,
                                     out: Optional[ExpertChoiceOut] = None,
                                     stream=None) -> ExpertChoiceOut:
    """The layer with expert-choice routing; see switch_moe_forward_expert_choice
    in include/switch_moe.h."""
    dev = x.device
    _contig(x, "x", None, dev)
    T, d, F, N = _layer_args(x, W_g, W1, W2, b_g, W1s, W2s, dev)
    p = make_params(T, d, F, N, capacity_factor, TOKEN_ORDER, gate_multiply, _dtype_code(x),
                    int(W1s is not None), expert_choice=1)
    if ws is None:
        ws = workspace(switch_moe_workspace_bytes(p), dev)
    C = switch_moe_capacity(T, N, capacity_factor) if T else 0
    if out is None:
        out = _ec_outputs(T, d, N, C, dev)
    want = (T * d, N * C, N * C, T, N, 1)
    for t, n, name in zip(out, want, ExpertChoiceOut._fields):
        if t.numel() != n or not t.is_contiguous():
            raise ValueError(f"out.{name} must be contiguous with {n} elements")
    with torch.cuda.device(dev):
        rc = _lib.switch_moe_forward_expert_choice(
            ctypes.byref(p), _ptr(x), _ptr(W_g), _ptr(b_g), _ptr(W1), _ptr(W2), _ptr(W1s),
            _ptr(W2s), _ptr(out.y), _ptr(out.chosen_token), _ptr(out.chosen_gate),
            _ptr(out.experts_per_token), _ptr(out.expert_counts), _ptr(out.aux_loss), _ptr(ws),
            ctypes.c_size_t(ws.numel()), _stream(stream))
    _check(rc, "switch_moe_forward_expert_choice")
    return out


def switch_moe_route_expert_choice(logits: torch.Tensor, capacity_factor: float,
                                   ws: Optional[torch.Tensor] = None,
                                   stream=None) -> ExpertChoiceOut:
    """Expert-choice routing on given fp32 logits [T, N] (y is None)."""
    dev = logits.device
    _contig(logits, "logits", torch.float32)
    T, N = logits.shape
    p = make_params(T, 8, 8, N, capacity_factor, TOKEN_ORDER, 1, F32, 0, expert_choice=1)
    if ws is None:
        ws = workspace(switch_moe_workspace_bytes(p), dev)
    C = switch_moe_capacity(T, N, capacity_factor) if T else 0
    o = _ec_outputs(T, None, N, C, dev)
    with torch.cuda.device(dev):
        rc = _lib.switch_moe_route_expert_choice(
            ctypes.byref(p), _ptr(logits), _ptr(o.chosen_token), _ptr(o.chosen_gate),
            _ptr(o.experts_per_token), _ptr(o.expert_counts), _ptr(o.aux_loss), _ptr(ws),
            ctypes.c_size_t(ws.numel()), _stream(stream))
    _check(rc, "switch_moe_route_expert_choice")
    return o


class BackwardOut(NamedTuple):
    dx: torch.Tensor                 # [T, d_model] fp32
    dW_g: torch.Tensor               # [N, d_model]
    db_g: Optional[torch.Tensor]     # [N] (None without b_g)
    dW1: torch.Tensor                # [N, d_ff, d_model]
    dW2: torch.Tensor                # [N, d_model, d_ff]
    dW1s: Optional[torch.Tensor]     # [d_ff, d_model] with a shared expert
    dW2s: Optional[torch.Tensor]     # [d_model, d_ff]


def switch_moe_backward_workspace_bytes(p: Params) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.switch_moe_backward_workspace_bytes(ctypes.byref(p), ctypes.byref(n)),
           "switch_moe_backward_workspace_bytes")
    return int(n.value)


def switch_moe_backward(x: torch.Tensor, W_g: torch.Tensor, W1: torch.Tensor, W2: torch.Tensor,
                        capacity_factor: float, fwd: ForwardOut, dy: torch.Tensor,
                        aux_coef: float = 0.0, priority_mode: int = TOKEN_ORDER,
                        gate_multiply: int = 1, b_g: Optional[torch.Tensor] = None,
                        W1s: Optional[torch.Tensor] = None, W2s: Optional[torch.Tensor] = None,
                        ws: Optional[torch.Tensor] = None, stream=None) -> BackwardOut:
    """Gradients of <dy, y> + aux_coef * L_aux for the forward that produced
    ``fwd`` (its routing outputs are reused); see switch_moe_backward in
    include/switch_moe.h."""
    dev = x.device
    _contig(x, "x", None, dev)
    _contig(dy, "dy", torch.float32, dev)
    T, d, F, N = _layer_args(x, W_g, W1, W2, b_g, W1s, W2s, dev)
    if dy.shape != (T, d):
        raise ValueError("dy must be [T, d_model]")
    for name, t, n in (("expert_id", fwd.expert_id, T), ("gate", fwd.gate, T),
                       ("slot", fwd.slot, T), ("expert_counts", fwd.expert_counts, N)):
        if t.numel() != n or not t.is_contiguous() or t.device != dev:
            raise ValueError(f"fwd.{name} must be a contiguous {n}-element tensor on {dev}")
    p = make_params(T, d, F, N, capacity_factor, priority_mode, gate_multiply, _dtype_code(x),
                    int(W1s is not None))
    if ws is None:
        ws = workspace(switch_moe_backward_workspace_bytes(p), dev)
    f32 = dict(dtype=torch.float32, device=dev)
    out = BackwardOut(torch.empty((T, d), **f32), torch.empty((N, d), **f32),
                      torch.empty(N, **f32) if b_g is not None else None,
                      torch.empty((N, F, d), **f32), torch.empty((N, d, F), **f32),
                      torch.empty((F, d), **f32) if W1s is not None else None,
                      torch.empty((d, F), **f32) if W1s is not None else None)
    with torch.cuda.device(dev):
        rc = _lib.switch_moe_backward(
            ctypes.byref(p), _ptr(x), _ptr(W_g), _ptr(b_g), _ptr(W1), _ptr(W2), _ptr(W1s),
            _ptr(W2s), _ptr(fwd.expert_id), _ptr(fwd.gate), _ptr(fwd.slot),
            _ptr(fwd.expert_counts), _ptr(dy), ctypes.c_float(aux_coef), _ptr(out.dx),
            _ptr(out.dW_g), _ptr(out.db_g), _ptr(out.dW1), _ptr(out.dW2), _ptr(out.dW1s),
            _ptr(out.dW2s), _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream))
    _check(rc, "switch_moe_backward")
    return out


def switch_moe_router_logits(x: torch.Tensor, W_g: torch.Tensor,
                             b_g: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """fp32 router logits [T, N] from the same device code the forward uses."""
    dev = x.device
    _contig(x, "x", None, dev)
    _contig(W_g, "W_g", torch.float32, dev)
    _contig(b_g, "b_g", torch.float32, dev)
    T, d = x.shape
    N = W_g.shape[0]
    p = make_params(T, d, 8, N, 1.0, TOKEN_ORDER, 1, _dtype_code(x), 0)
    ws = workspace(switch_moe_workspace_bytes(p), dev)
    logits = torch.empty((T, N), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        rc = _lib.switch_moe_router_logits(ctypes.byref(p), _ptr(x), _ptr(W_g), _ptr(b_g),
                                           _ptr(logits), _ptr(ws), ctypes.c_size_t(ws.numel()),
                                           _stream(stream))
    _check(rc, "switch_moe_router_logits")
    return logits


def switch_moe_selftest_wait_timeout(timeout_ns: int = 20_000_000, stream=None) -> None:
    """Enqueue the diagnostic kernel whose bounded wait is bound to expire."""
    _check(_lib.switch_moe_selftest_wait_timeout(int(timeout_ns), _stream(stream)),
           "switch_moe_selftest_wait_timeout")


def switch_moe_set_phase_events(events) -> None:
    """events: a list of NUM_PHASE_EVENTS torch.cuda.Event(enable_timing=True)
    (recorded once so that they own a CUDA event), or None to stop."""
    if events is None:
        _check(_lib.switch_moe_set_phase_events(None, NUM_PHASE_EVENTS),
               "switch_moe_set_phase_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(_lib.switch_moe_set_phase_events(arr, len(events)), "switch_moe_set_phase_events")


def switch_moe_sync_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status word."""
    return int(_lib.switch_moe_sync_status(_stream(stream)))
