"""Top-2 token choice on the CUDA path against the oracle (the variant set
beside Switch's top-1 in "Top-1 路由 (Top-1 Routing)", compassingai.com,
industry-position and comparison sections; the gate-weighted sum over the
chosen set of the Switch Transformer walk-through's Switch-layer section;
Mixtral's softmax over the top-k in "Which Routing Does Each MoE Model Use?").

* routing on given fp32 logits: the chosen pair, slots, drops and
  expert_counts bit-exact against the oracle's definition on the same
  logits; gates within fp32 softmax rounding; aux_loss within 1e-5 relative;
* the forward end to end: routing bit-exact against the oracle applied to
  the kernel's own fp32 logits (switch_moe_router_logits, which the forward
  routes on bit for bit), y within max|dy| / rms <= 1e-2 on every token;
  cases cover both tensor-core router epilogues (N <= 128 and N > 128), the
  one-launch FFN, token tiles of 256 (separate GEMMs), the K-split second
  GEMM with the combine kernel, fp32 layers and the shared expert;
* argument checks and workspace sizes on the host.
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import AUX_TOL, GATE_RTOL, Y_TOL, np_
from workloads import Workload, make_inputs


def _logits(T, N, seed, kind):
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        return torch.randn(T, N, generator=g).float() * 2.0
    if kind == "ints":          # many exact ties between the first and second choice
        return torch.randint(-2, 3, (T, N), generator=g).float()
    if kind == "equal":
        return torch.zeros(T, N)
    if kind == "skew":          # Zipf-biased: hot experts overflow
        z = torch.tensor([(e + 1) ** -1.1 for e in range(N)], dtype=torch.float64)
        b = 0.6 * torch.log(z / z.sum())
        return (torch.randn(T, N, generator=g, dtype=torch.float64) * 0.55 + b).float()
    raise ValueError(kind)


def _oracle_top2(logits32, N, C, renorm):
    l = logits32.double().numpy()
    c = oracle.candidates(l, 2)
    p = oracle.softmax(l)
    slot, drop, _ = oracle.assign_slots_top2(c, N, C)
    return c, oracle.top2_gates(p, c, renorm), slot, drop, np.bincount(c[:, 0], minlength=N), p


ROUTE_CASES = [
    # T, N, cf, renormalize, kind
    (8192, 128, 1.25, 0, "skew"),
    (8192, 128, 2.5, 1, "skew"),
    (16384, 64, 1.0, 1, "skew"),
    (777, 5, 0.7, 0, "normal"),
    (1000, 7, 0.5, 1, "ints"),
    (300, 4, 1.0, 0, "equal"),       # every token picks experts 0 and 1
    (64, 2, 2.0, 1, "normal"),       # N = 2: every token uses both experts
    (2048, 256, 0.5, 0, "normal"),
    (33, 1024, 4.0, 1, "normal"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("T,N,cf,rn,kind", ROUTE_CASES)
def test_route_top2_matches_oracle(lib, T, N, cf, rn, kind):
    logits = _logits(T, N, T * 31 + N + rn, kind)
    gpu = lib.switch_moe_route_from_logits(logits.cuda(), cf, 0, top_k=2, renormalize=rn)
    assert lib.switch_moe_sync_status() == 0
    C = oracle.capacity(T, N, cf)
    c, g, s, d, counts, p = _oracle_top2(logits, N, C, rn)
    assert tuple(gpu.expert_id.shape) == (T, 2)
    assert np.array_equal(np_(gpu.expert_id), c)
    assert np.array_equal(np_(gpu.slot), s)
    assert np.array_equal(np_(gpu.drop_mask), d)
    assert np.array_equal(np_(gpu.expert_counts), counts)     # choice 0 only
    np.testing.assert_allclose(np_(gpu.gate).astype(np.float64), g, rtol=4 * GATE_RTOL, atol=0)
    aux = oracle.aux_loss(p, counts)
    assert abs(float(np_(gpu.aux_loss)[0]) - aux) <= AUX_TOL * abs(aux)
    # choice 0 is exactly the top-1 routing of the same logits
    plain = lib.switch_moe_route_from_logits(logits.cuda(), cf, 0)
    assert np.array_equal(np_(gpu.slot)[:, 0], np_(plain.slot))


FWD_CASES = [
    # name, T, d, F, N, cf, dtype, renormalize, shared, Zipf strength of the logit bias
    ("bf16-ffn", 4096, 256, 512, 32, 1.5, "bf16", 0, 0, 0.6),
    ("bf16-ffn-renorm", 4096, 256, 512, 32, 1.0, "bf16", 1, 0, 0.6),
    ("bf16-N200-tmem-router", 2048, 128, 256, 200, 2.0, "bf16", 1, 0, 0.3),
    ("bf16-shared", 1000, 128, 256, 8, 1.2, "bf16", 1, 1, 0.6),
    ("f32", 512, 64, 256, 8, 1.0, "f32", 0, 0, 1.5),
    ("f32-shared", 300, 64, 128, 4, 1.5, "f32", 1, 1, 0.6),
    ("bf16-big-C", 3000, 128, 256, 4, 1.2, "bf16", 0, 0, 0.6),          # token tiles of 256
    ("bf16-decode", 64, 512, 1024, 8, 2.0, "bf16", 1, 0, 0.6),      # 16-token tiles
    ("bf16-ksplit", 300, 512, 1024, 2, 1.0, "bf16", 1, 0, 0.0),     # C = 150: K-split GEMM 2
    ("bf16-one-token", 1, 64, 128, 4, 1.0, "bf16", 1, 0, 0.0),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", FWD_CASES, ids=[c[0] for c in FWD_CASES])
def test_forward_top2(lib, case):
    name, T, d, F, N, cf, dt, rn, sh, lam = case
    w = Workload(name, T, d, F, N, cf, dt, 0.3, has_shared=sh, zipf_s=1.1, zipf_lambda=lam)
    inp = make_inputs(w, seed=13, device="cuda")
    out = lib.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, cf, b_g=inp.b_g,
                                 W1s=inp.W1s, W2s=inp.W2s, top_k=2, renormalize=rn)
    lg = lib.switch_moe_router_logits(inp.x, inp.W_g, inp.b_g)   # what the forward routed on
    assert lib.switch_moe_sync_status() == 0
    C = oracle.capacity(T, N, cf)
    c, g, s, dr, counts, _ = _oracle_top2(lg.cpu(), N, C, rn)
    assert np.array_equal(np_(out.expert_id), c)
    assert np.array_equal(np_(out.slot), s)
    assert np.array_equal(np_(out.drop_mask), dr)
    assert np.array_equal(np_(out.expert_counts), counts)
    np.testing.assert_allclose(np_(out.gate).astype(np.float64), g, rtol=4 * GATE_RTOL, atol=0)
    getter = lambda i: (inp.W1[i].cpu(), inp.W2[i].cpu())  # noqa: E731
    y_ref = oracle.forward_rows_top2(np.arange(T), inp.x.cpu(), c, g, s, 1, getter,
                                     None if inp.W1s is None else inp.W1s.cpu(),
                                     None if inp.W2s is None else inp.W2s.cpu())
    rms = np.sqrt((y_ref ** 2).mean())
    err = np.abs(np_(out.y).astype(np.float64) - y_ref).max() / rms
    assert err <= Y_TOL, f"y max|err|/rms = {err:.3g}"
    if T > 1:
        both = (dr == 0).all(axis=1)
        assert both.sum() > 0 and (dr[:, 1] == 1).sum() > 0, "the shape should keep and drop"


@pytest.mark.gpu
def test_forward_top2_oracle_end_to_end(lib):
    """A small layer run whole through the oracle's own top-2 forward."""
    w = Workload("e2e", 256, 64, 128, 8, 1.0, "bf16", 0.3, zipf_s=1.1, zipf_lambda=0.6)
    inp = make_inputs(w, seed=17, device="cuda")
    out = lib.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, 1.0, b_g=inp.b_g, top_k=2)
    assert lib.switch_moe_sync_status() == 0
    ref = oracle.forward_top2(inp.x.cpu(), inp.W_g.cpu(), inp.W1.cpu(), inp.W2.cpu(), 1.0,
                              b_g=inp.b_g.cpu() if inp.b_g is not None else None)
    lg = ref["logits"]
    top3 = np.sort(lg, axis=1)[:, -3:]
    clear = ((top3[:, 2] - top3[:, 1]) > 1e-5) & ((top3[:, 1] - top3[:, 0]) > 1e-5)
    assert clear.all(), "seeded inputs are free of near-ties"
    assert np.array_equal(np_(out.expert_id), ref["expert_id"])
    assert np.array_equal(np_(out.slot), ref["slot"])
    rms = np.sqrt((ref["y"] ** 2).mean())
    assert np.abs(np_(out.y).astype(np.float64) - ref["y"]).max() / rms <= Y_TOL
    assert abs(float(np_(out.aux_loss)[0]) - ref["aux_loss"]) <= AUX_TOL * ref["aux_loss"]


@pytest.mark.gpu
def test_top_k_one_is_plain_top1(lib):
    w = Workload("k1", 2048, 128, 256, 16, 0.8, "bf16", 0.3, zipf_s=1.1, zipf_lambda=0.6)
    inp = make_inputs(w, seed=5, device="cuda")
    a = lib.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, 0.8, b_g=inp.b_g)
    b = lib.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, 0.8, b_g=inp.b_g, top_k=1)
    assert lib.switch_moe_sync_status() == 0
    for f in a._fields:
        assert torch.equal(getattr(a, f), getattr(b, f)), f


@pytest.mark.gpu
def test_top2_hostio_matches_device(lib):
    w = Workload("hio", 1024, 128, 256, 16, 1.0, "bf16", 0.3, zipf_s=1.1, zipf_lambda=0.6)
    inp = make_inputs(w, seed=7, device="cuda")
    a = lib.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, 1.0, b_g=inp.b_g, top_k=2,
                               renormalize=1)
    b = lib.switch_moe_forward_hostio(inp.x.cpu(), inp.W_g, inp.W1, inp.W2, 1.0, b_g=inp.b_g,
                                      top_k=2, renormalize=1)
    torch.cuda.synchronize()
    assert lib.switch_moe_sync_status() == 0
    for f in ("expert_id", "gate", "slot", "drop_mask", "expert_counts"):
        assert torch.equal(getattr(a, f).cpu(), getattr(b, f)), f
    # the two adds into a row commute exactly (no shared expert): y is identical
    assert torch.equal(a.y.cpu(), b.y)


@pytest.mark.parametrize("kw,code", [
    (dict(top_k=3), "INVALID_ARG"), (dict(top_k=-1), "INVALID_ARG"),
    (dict(renormalize=1), "INVALID_ARG"), (dict(top_k=2, renormalize=2), "INVALID_ARG"),
    (dict(top_k=2, priority_mode=1), "UNSUPPORTED"), (dict(top_k=2, N=1), "UNSUPPORTED"),
    (dict(top_k=2, expand=2), "UNSUPPORTED"),
])
def test_top2_argument_checks(kw, code):
    from switch_top_expert_router_b300 import build
    build.build()
    import switch_top_expert_router_b300 as sm
    args = dict(T=1000, d_model=64, d_ff=128, N=8, capacity_factor=1.0, priority_mode=0,
                gate_multiply=1, dtype=1, has_shared=0)
    args.update(kw)
    with pytest.raises(sm.SwitchMoEError) as ei:
        sm.switch_moe_workspace_bytes(sm.make_params(**args))
    assert ei.value.code == getattr(sm, "SWITCH_MOE_ERR_" + code)


def test_top2_workspace_and_hostio_sizes():
    from switch_top_expert_router_b300 import build
    build.build()
    import switch_top_expert_router_b300 as sm
    T, N = 1000, 8
    p1 = sm.make_params(T, 64, 128, N, 1.0)
    p2 = sm.make_params(T, 64, 128, N, 1.0, top_k=2, renormalize=1)
    w1, w2 = sm.switch_moe_workspace_bytes(p1), sm.switch_moe_workspace_bytes(p2)
    assert w2 > w1
    h1, h2 = sm.switch_moe_hostio_workspace_bytes(p1), sm.switch_moe_hostio_workspace_bytes(p2)
    # the host-IO region holds [T, 2] copies of the four per-token outputs
    assert (h2 - w2) - (h1 - w1) >= T * (4 + 4 + 4 + 1)
