"""Seeded synthetic inputs for the Switch top-1 MoE layer.

This module draws random tensors and nothing else: it holds none of the
layer's arithmetic (no routing, capacity, FFN or loss). Both the CUDA path
and the CPU oracle consume exactly the tensors it returns, so the two sides
see identical bf16 / fp32 values.

Shapes and distributions follow the five layer shapes the library is
measured on (tokens T, model width d, FFN width F, routed experts N,
capacity factor cf):

=========  =====  ====  =====  ===  ====  ========  ==============================
name         T     d      F     N    cf   dtype     structure
=========  =====  ====  =====  ===  ====  ========  ==============================
tiny        512    64    256    8   1.0   fp32      W_g ~ N(0, 0.1^2)
base       8192   768   3072  128   1.25  bf16      uniform-ish routing
skew      16384  1024   4096   64   1.0   bf16      Zipf(1.1) logit bias, gate prio
wide       4096  5120   8192  128   1.25  bf16      + one always-on shared expert
decode       64  4096  14336    8   2.0   bf16      weight-bound (few tokens)
=========  =====  ====  =====  ===  ====  ========  ==============================

x ~ N(0, 1); W_g ~ N(0, sigma_g^2) in fp32 (the router is always fp32);
W1 ~ N(0, 1/d) and W2 ~ N(0, 1/F) (fan-in scaling), drawn in fp32 and cast
once to the layer dtype.  Each tensor has its own seed, derived from the
workload seed, and each expert's weights have their own seed, so a sample of
experts can be regenerated without materialising the rest.

The "Base" shape is the Switch-Base layer of the Switch Transformer
walk-through (personwebsite.pages.dev/moe-switch, Table 1: d_model 768,
d_ff 3072, 128 experts at capacity factor 1.0-1.25); the pages measure on
C4 / mT5 text, which these seeded Gaussian inputs stand in for: a layer
forward depends only on shapes and value distributions.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["Workload", "CONFIGS", "make_inputs", "expert_weights", "Inputs"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d_model: int
    d_ff: int
    N: int
    capacity_factor: float
    dtype: str                  # "f32" or "bf16": dtype of x, W1, W2 (and W1s, W2s)
    router_std: float           # std of W_g entries
    priority_mode: int = 0      # 0 = token order, 1 = gate-value priority
    gate_multiply: int = 1
    has_shared: int = 0
    zipf_s: float = 0.0         # >0: add lam * ln z_e to logit e, z_e ~ (e+1)^-s
    zipf_lambda: float = 0.0

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# Zipf strength for the skewed-overflow shape.  Frozen from
# workloads/calibrate_skew.py, which runs the oracle's router and slot
# assignment on the seed-0 inputs and reports the drop fraction (the shape
# asks for 10-30 % of tokens to overflow; this value gives about 19 %).
SKEW_ZIPF_LAMBDA = 0.12

CONFIGS = {
    "tiny": Workload("tiny", 512, 64, 256, 8, 1.0, "f32", 0.1),
    "base": Workload("base", 8192, 768, 3072, 128, 1.25, "bf16", 0.02),
    "skew": Workload("skew", 16384, 1024, 4096, 64, 1.0, "bf16", 0.02,
                     priority_mode=1, zipf_s=1.1, zipf_lambda=SKEW_ZIPF_LAMBDA),
    "wide": Workload("wide", 4096, 5120, 8192, 128, 1.25, "bf16", 0.02,
                     has_shared=1),
    "decode": Workload("decode", 64, 4096, 14336, 8, 2.0, "bf16", 0.02),
}

# tensor ids for seed derivation
_ID_X, _ID_WG, _ID_W1, _ID_W2, _ID_W1S, _ID_W2S = 1, 2, 3, 4, 5, 6


def _seed(seed: int, tensor_id: int, sub: int = 0) -> int:
    return (seed * 1000003 + tensor_id * 7919 + sub * 104729) & 0x7FFFFFFFFFFF


def _randn(shape, seed: int, device, std: float = 1.0) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def zipf_bias(w: Workload) -> Optional[torch.Tensor]:
    """Per-expert logit offsets lam * ln z_e with z_e proportional to (e+1)^-s
    (normalised), or None when the workload has no skew."""
    if w.zipf_s <= 0:
        return None
    z = [(e + 1) ** (-w.zipf_s) for e in range(w.N)]
    tot = sum(z)
    return torch.tensor([w.zipf_lambda * math.log(v / tot) for v in z],
                        dtype=torch.float32)


def expert_weights(w: Workload, e: int, seed: int = 0, device="cpu"):
    """(W1_e [F, d], W2_e [d, F]) of routed expert e, or of the shared expert
    when e == -1, in the workload dtype."""
    if e < 0:
        i1, i2, sub = _ID_W1S, _ID_W2S, 0
    else:
        i1, i2, sub = _ID_W1, _ID_W2, e
    W1 = _randn((w.d_ff, w.d_model), _seed(seed, i1, sub), device,
                1.0 / math.sqrt(w.d_model)).to(w.torch_dtype)
    W2 = _randn((w.d_model, w.d_ff), _seed(seed, i2, sub), device,
                1.0 / math.sqrt(w.d_ff)).to(w.torch_dtype)
    return W1, W2


@dataclasses.dataclass
class Inputs:
    x: torch.Tensor                 # [T, d]        layer dtype
    W_g: torch.Tensor               # [N, d]        fp32
    b_g: Optional[torch.Tensor]     # [N] fp32 or None
    W1: torch.Tensor                # [N, F, d]     layer dtype
    W2: torch.Tensor                # [N, d, F]     layer dtype
    W1s: Optional[torch.Tensor]     # [F, d] or None
    W2s: Optional[torch.Tensor]     # [d, F] or None


def make_inputs(w: Workload, seed: int = 0, device="cpu",
                with_experts: bool = True) -> Inputs:
    """Draw every input of workload ``w`` on ``device``.

    ``with_experts=False`` skips the routed expert weights (W1/W2 are then
    empty tensors); callers regenerate single experts with
    :func:`expert_weights`."""
    x = _randn((w.T, w.d_model), _seed(seed, _ID_X), device).to(w.torch_dtype)
    W_g = _randn((w.N, w.d_model), _seed(seed, _ID_WG), device, w.router_std)
    b = zipf_bias(w)
    b_g = b.to(device) if b is not None else None
    if with_experts:
        W1 = torch.empty((w.N, w.d_ff, w.d_model), dtype=w.torch_dtype, device=device)
        W2 = torch.empty((w.N, w.d_model, w.d_ff), dtype=w.torch_dtype, device=device)
        for e in range(w.N):
            a, b2 = expert_weights(w, e, seed, device)
            W1[e].copy_(a)
            W2[e].copy_(b2)
    else:
        W1 = torch.empty((0,), dtype=w.torch_dtype, device=device)
        W2 = torch.empty((0,), dtype=w.torch_dtype, device=device)
    W1s = W2s = None
    if w.has_shared:
        W1s, W2s = expert_weights(w, -1, seed, device)
    return Inputs(x, W_g, b_g, W1, W2, W1s, W2s)
