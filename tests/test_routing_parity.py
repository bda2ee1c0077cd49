"""Routing parity: switch_moe_route_from_logits (CUDA) vs the oracle on the
same fp32 logits -- expert_id, slot, drop_mask and expert_counts bit-exact,
gate within fp32 rounding, aux_loss within 1e-5 relative."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import check_routing_same_logits, np_

pytestmark = pytest.mark.gpu


def _logits(T, N, seed, kind="normal", scale=1.0):
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        return (torch.randn(T, N, generator=g) * scale).float()
    if kind == "ints":          # many exact ties
        return torch.randint(-2, 3, (T, N), generator=g).float()
    if kind == "equal":
        return torch.zeros(T, N)
    if kind == "dup_rows":      # identical tokens -> identical gates (gate-priority ties)
        row = torch.randn(1, N, generator=g)
        return row.repeat(T, 1).float()
    if kind == "skew":
        z = torch.tensor([(e + 1) ** -1.1 for e in range(N)], dtype=torch.float64)
        return (torch.randn(T, N, generator=g) * 0.55 + 0.12 * torch.log(z / z.sum())).float()
    raise ValueError(kind)


CASES = [
    # T, N, cf, mode, kind
    (512, 8, 1.0, 0, "normal"),        # tiny layer shape
    (8192, 128, 1.25, 0, "normal"),    # Switch-Base shape
    (16384, 64, 1.0, 1, "skew"),       # skewed overflow, gate priority
    (4096, 128, 1.25, 0, "normal"),    # wide shape
    (64, 8, 2.0, 0, "normal"),         # decode shape
    (1000, 7, 1.0, 0, "ints"),         # ragged T, ties
    (1000, 7, 1.0, 1, "ints"),
    (999, 3, 0.3, 1, "normal"),        # heavy overflow, gate priority
    (333, 5, 1.0, 0, "equal"),         # all ties -> expert 0, first C kept
    (333, 5, 1.0, 1, "equal"),
    (300, 4, 1.0, 1, "dup_rows"),      # equal gates: token order breaks ties
    (1, 1, 1.0, 0, "normal"),          # one token, one expert
    (77, 1, 1.0, 1, "normal"),         # N = 1
    (2048, 1024, 1.0, 0, "normal"),    # N at its maximum
    (5000, 16, 16.0, 0, "normal"),     # cf >= N: nothing dropped
    (5000, 16, 0.01, 1, "normal"),     # C = 4
    (20000, 1, 0.5, 1, "normal"),      # more tokens than one shared-memory sort: radix select
    (40000, 2, 0.3, 1, "skew"),        # same, two experts
]


@pytest.mark.parametrize("T,N,cf,mode,kind", CASES)
def test_route_from_logits_matches_oracle(lib, T, N, cf, mode, kind):
    logits = _logits(T, N, seed=T * 31 + N, kind=kind, scale=2.0)
    gpu = lib.switch_moe_route_from_logits(logits.cuda(), cf, mode)
    assert lib.switch_moe_sync_status() == 0
    C = oracle.capacity(T, N, cf)
    info = check_routing_same_logits(gpu, logits, N, C, mode)
    if kind == "equal":
        assert np.all(np_(gpu.expert_id) == 0)
        assert np.array_equal(np_(gpu.slot)[:C], np.arange(min(C, T)))
        assert np.all(np_(gpu.slot)[C:] == -1)
        assert float(np_(gpu.aux_loss)[0]) == pytest.approx(1.0, abs=1e-6)
    if cf >= N:
        assert np_(gpu.drop_mask).sum() == 0
    assert info["counts"].sum() == T


def test_route_is_deterministic(lib):
    logits = _logits(8192, 128, 3).cuda()
    a = lib.switch_moe_route_from_logits(logits, 1.0, 1)
    b = lib.switch_moe_route_from_logits(logits, 1.0, 1)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_empty_batch(lib):
    logits = torch.empty((0, 8), device="cuda")
    o = lib.switch_moe_route_from_logits(logits, 1.0, 0)
    assert lib.switch_moe_sync_status() == 0
    assert np.all(np_(o.expert_counts) == 0) and float(np_(o.aux_loss)[0]) == 0.0
