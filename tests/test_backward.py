"""Backward of the top-1 layer on the CUDA path against the oracle's
backward (pinned by central differences of the pinned forward).

The CUDA backward recomputes the forward's intermediates in fp32 from the
exact inputs and reuses the forward's routing; the oracle runs the same
definition in fp64 with its own routing, so the seeded inputs are checked
to be free of near-ties first (the routing then agrees).  Every gradient
must match within max|d| / rms(ref) <= 1e-4 (fp32 accumulation over at
most a few thousand terms against fp64).
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import np_
from workloads import Workload, make_inputs

GRAD_TOL = 1e-4

CASES = [
    # name, T, d, F, N, cf, dtype, mode, gate_multiply, shared, aux_coef, zipf strength
    ("f32", 256, 64, 128, 8, 1.0, "f32", 0, 1, 0, 0.01, 0.6),
    ("bf16", 512, 128, 256, 8, 1.0, "bf16", 0, 1, 0, 0.01, 0.6),
    ("bf16-gate-priority", 512, 128, 256, 8, 0.8, "bf16", 1, 1, 0, 0.05, 0.6),
    ("bf16-no-gate-mul", 300, 64, 128, 4, 1.0, "bf16", 0, 0, 0, 0.02, 0.6),
    ("bf16-shared", 300, 64, 192, 4, 1.0, "bf16", 0, 1, 1, 0.0, 0.6),
    ("bf16-ragged", 333, 72, 136, 5, 0.7, "bf16", 0, 1, 0, 0.1, 0.3),
    ("bf16-one-expert", 64, 64, 128, 1, 1.0, "bf16", 0, 1, 0, 0.5, 0.0),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_oracle(lib, case):
    name, T, d, F, N, cf, dt, mode, gm, sh, alpha, lam = case
    w = Workload(name, T, d, F, N, cf, dt, 0.3, has_shared=sh, zipf_s=1.1, zipf_lambda=lam)
    inp = make_inputs(w, seed=23, device="cuda")
    dy = torch.randn(T, d, generator=torch.Generator().manual_seed(T + d)).cuda()
    fwd = lib.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, cf, mode, gm, b_g=inp.b_g,
                                 W1s=inp.W1s, W2s=inp.W2s)
    got = lib.switch_moe_backward(inp.x, inp.W_g, inp.W1, inp.W2, cf, fwd, dy, aux_coef=alpha,
                                  priority_mode=mode, gate_multiply=gm, b_g=inp.b_g,
                                  W1s=inp.W1s, W2s=inp.W2s)
    torch.cuda.synchronize()
    assert lib.switch_moe_sync_status() == 0
    cpu = lambda t: None if t is None else t.cpu()  # noqa: E731
    ref = oracle.backward(cpu(inp.x), cpu(inp.W_g), cpu(inp.W1), cpu(inp.W2), cf, cpu(dy),
                          mode, gm, cpu(inp.b_g), cpu(inp.W1s), cpu(inp.W2s), aux_coef=alpha)
    f = ref["forward"]
    top2 = np.sort(f["logits"], axis=1)[:, -2:] if N > 1 else None
    if top2 is not None:
        assert (top2[:, 1] - top2[:, 0]).min() > 1e-5, "seeded inputs have a near-tie"
    assert np.array_equal(np_(fwd.expert_id), f["expert_id"])
    assert np.array_equal(np_(fwd.slot), f["slot"])
    pairs = [("dx", got.dx, ref["dx"]), ("dW_g", got.dW_g, ref["dW_g"]),
             ("dW1", got.dW1, ref["dW1"]), ("dW2", got.dW2, ref["dW2"])]
    if inp.b_g is not None:
        pairs.append(("db_g", got.db_g, ref["db_g"]))
    if sh:
        pairs += [("dW1s", got.dW1s, ref["dW1s"]), ("dW2s", got.dW2s, ref["dW2s"])]
    for nm, g, r in pairs:
        g = np_(g).astype(np.float64)
        rms = np.sqrt((r ** 2).mean())
        if rms == 0:
            assert np.abs(g).max() == 0, nm
            continue
        err = np.abs(g - r).max() / rms
        assert err <= GRAD_TOL, f"{name}: {nm} max|d|/rms = {err:.3g}"


@pytest.mark.gpu
def test_backward_gradient_descent_lowers_the_loss(lib):
    """A small step of the expert weights against the CUDA gradient lowers
    <dy, y> as computed by the CUDA forward, by step * |grad|^2 to first
    order (the routing depends on W_g alone and does not move)."""
    w = Workload("gd", 512, 128, 256, 8, 1.0, "f32", 0.3, zipf_s=1.1, zipf_lambda=0.6)
    inp = make_inputs(w, seed=29, device="cuda")
    dy = torch.randn(512, 128, generator=torch.Generator().manual_seed(3)).cuda()

    def loss(W1, W2):
        f = lib.switch_moe_forward(inp.x, inp.W_g, W1, W2, 1.0, b_g=inp.b_g)
        return float((f.y.double() * dy.double()).sum()), f

    l0, f0 = loss(inp.W1, inp.W2)
    g = lib.switch_moe_backward(inp.x, inp.W_g, inp.W1, inp.W2, 1.0, f0, dy, b_g=inp.b_g)
    step = 1e-4
    l1, f1 = loss(inp.W1 - step * g.dW1, inp.W2 - step * g.dW2)
    assert torch.equal(f1.expert_id, f0.expert_id) and torch.equal(f1.slot, f0.slot)
    gn2 = float((g.dW1.double() ** 2).sum() + (g.dW2.double() ** 2).sum())
    assert l1 < l0
    assert abs((l0 - l1) - step * gn2) <= 0.05 * step * gn2


def test_backward_argument_checks():
    from switch_top_expert_router_b300 import build
    build.build()
    import switch_top_expert_router_b300 as sm
    for kw in (dict(top_k=2), dict(expand=2), dict(expert_choice=1)):
        p = sm.make_params(512, 64, 128, 8, 1.0, **kw)
        with pytest.raises(sm.SwitchMoEError) as ei:
            sm.switch_moe_backward_workspace_bytes(p)
        assert ei.value.code == sm.SWITCH_MOE_ERR_UNSUPPORTED
    p = sm.make_params(8192, 768, 3072, 128, 1.25)
    # fp32 slots rows and hidden activations: at least 4 [N C, d] + 2 [N C, F]
    assert sm.switch_moe_backward_workspace_bytes(p) >= 4 * 128 * 80 * (2 * 768 + 3072)
