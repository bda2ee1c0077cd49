"""Expanded Drop (the tokens an over-full expert drops take a free slot of
their next candidate expert; "MoE 专家容量因子与 Token 丢弃", wiblog.cn,
inference section) on the CUDA path against the oracle.

* routing on given fp32 logits: expert, slot, drop and expert_counts
  bit-exact against the oracle's definition on the same logits, gates within
  fp32 softmax rounding, aux_loss within 1e-5 relative;
* the forward end to end: routing bit-exact against the oracle applied to
  the kernel's own fp32 logits (the ones switch_moe_router_logits returns,
  which the forward routes on bit for bit), y within max|dy| / rms <= 1e-2;
* expand = 1 is the plain top-1 path; argument checks on the host.
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import AUX_TOL, GATE_RTOL, Y_TOL, np_
from workloads import Workload, expert_weights, make_inputs


def _logits(T, N, seed, kind):
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        return torch.randn(T, N, generator=g).float() * 2.0
    if kind == "ints":          # many exact ties, also among later candidates
        return torch.randint(-2, 3, (T, N), generator=g).float()
    if kind == "equal":
        return torch.zeros(T, N)
    if kind == "skew":          # Zipf-biased: hot experts overflow
        z = torch.tensor([(e + 1) ** -1.1 for e in range(N)], dtype=torch.float64)
        b = 0.6 * torch.log(z / z.sum())
        return (torch.randn(T, N, generator=g, dtype=torch.float64) * 0.55 + b).float()
    raise ValueError(kind)


def _oracle_expanded(logits32, N, C, k):
    l = logits32.double().numpy()
    e, s, d, used = oracle.assign_slots_expanded(oracle.candidates(l, k), N, C)
    p = oracle.softmax(l)
    return e, s, d, used, p[np.arange(l.shape[0]), e], np.bincount(np.argmax(l, axis=1),
                                                                     minlength=N)


ROUTE_CASES = [
    # T, N, cf, k, kind
    (8192, 128, 1.0, 2, "skew"),
    (8192, 128, 1.0, 4, "skew"),
    (16384, 64, 1.0, 3, "skew"),
    (777, 5, 0.7, 3, "normal"),
    (1000, 7, 0.5, 2, "ints"),
    (1000, 7, 0.5, 4, "ints"),
    (300, 4, 1.0, 4, "equal"),       # everything on expert 0 first, then 1, 2, 3
    (64, 8, 2.0, 2, "normal"),
    (2048, 256, 0.5, 2, "normal"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("T,N,cf,k,kind", ROUTE_CASES)
def test_route_expanded_matches_oracle(lib, T, N, cf, k, kind):
    logits = _logits(T, N, T * 17 + N + k, kind)
    gpu = lib.switch_moe_route_from_logits(logits.cuda(), cf, 0, expand=k)
    assert lib.switch_moe_sync_status() == 0
    C = oracle.capacity(T, N, cf)
    e, s, d, used, g, counts = _oracle_expanded(logits, N, C, k)
    assert np.array_equal(np_(gpu.expert_id), e)
    assert np.array_equal(np_(gpu.slot), s)
    assert np.array_equal(np_(gpu.drop_mask), d)
    assert np.array_equal(np_(gpu.expert_counts), counts)     # top-1 counts, not the fills
    np.testing.assert_allclose(np_(gpu.gate).astype(np.float64), g, rtol=GATE_RTOL, atol=0)
    ref = oracle.route_from_logits(logits)
    aux = oracle.aux_loss(ref["probs"], counts)
    assert abs(float(np_(gpu.aux_loss)[0]) - aux) <= AUX_TOL * abs(aux)
    plain = lib.switch_moe_route_from_logits(logits.cuda(), cf, 0)
    assert int(np_(gpu.drop_mask).sum()) <= int(np_(plain.drop_mask).sum())


FWD_CASES = [
    # name, T, d, F, N, cf, dtype, k, shared, Zipf strength of the logit bias
    # (strong enough that hot experts overflow while cold ones have room)
    ("bf16-skew-k2", 4096, 256, 512, 32, 1.0, "bf16", 2, 0, 0.6),
    ("bf16-skew-k4", 4096, 256, 512, 32, 1.0, "bf16", 4, 0, 0.6),
    ("bf16-shared-k3", 1000, 128, 256, 8, 0.8, "bf16", 3, 1, 0.6),
    ("f32-k2", 512, 64, 256, 8, 0.6, "f32", 2, 0, 1.5),
    ("bf16-big-C-k2", 3000, 128, 256, 4, 0.9, "bf16", 2, 0, 0.6),      # token tiles of 256
    ("bf16-decode-k2", 64, 512, 1024, 8, 0.9, "bf16", 2, 0, 0.6),   # 16-token tiles
    ("bf16-ksplit-k2", 300, 512, 1024, 2, 1.0, "bf16", 2, 0, 1.5),  # C = 150: K-split GEMM 2
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", FWD_CASES, ids=[c[0] for c in FWD_CASES])
def test_forward_expanded(lib, case):
    name, T, d, F, N, cf, dt, k, sh, lam = case
    w = Workload(name, T, d, F, N, cf, dt, 0.3, has_shared=sh, zipf_s=1.1, zipf_lambda=lam)
    inp = make_inputs(w, seed=11, device="cuda")
    out = lib.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, cf, b_g=inp.b_g,
                                 W1s=inp.W1s, W2s=inp.W2s, expand=k)
    lg = lib.switch_moe_router_logits(inp.x, inp.W_g, inp.b_g)   # what the forward routed on
    assert lib.switch_moe_sync_status() == 0
    C = oracle.capacity(T, N, cf)
    e, s, dr, used, g, counts = _oracle_expanded(lg.cpu(), N, C, k)
    assert np.array_equal(np_(out.expert_id), e)
    assert np.array_equal(np_(out.slot), s)
    assert np.array_equal(np_(out.drop_mask), dr)
    assert np.array_equal(np_(out.expert_counts), counts)
    np.testing.assert_allclose(np_(out.gate).astype(np.float64), g, rtol=GATE_RTOL, atol=0)
    # y of every token with these routing decisions, in fp64
    getter = lambda i: (inp.W1[i].cpu(), inp.W2[i].cpu())  # noqa: E731
    y_ref = oracle.forward_rows(np.arange(T), inp.x.cpu(), e, g, s, 1, getter,
                                None if inp.W1s is None else inp.W1s.cpu(),
                                None if inp.W2s is None else inp.W2s.cpu())
    rms = np.sqrt((y_ref ** 2).mean())
    err = np.abs(np_(out.y).astype(np.float64) - y_ref).max() / rms
    assert err <= Y_TOL, f"y max|err|/rms = {err:.3g}"
    plain = lib.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, cf, b_g=inp.b_g,
                                   W1s=inp.W1s, W2s=inp.W2s)
    assert lib.switch_moe_sync_status() == 0
    moved = (np_(plain.drop_mask) == 1) & (np_(out.drop_mask) == 0)
    assert moved.sum() > 0, "the shape should re-route some overflow"


@pytest.mark.gpu
def test_expand_one_is_plain_top1(lib):
    w = Workload("k1", 2048, 128, 256, 16, 0.8, "bf16", 0.3, zipf_s=1.1, zipf_lambda=0.6)
    inp = make_inputs(w, seed=5, device="cuda")
    a = lib.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, 0.8, b_g=inp.b_g)
    b = lib.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, 0.8, b_g=inp.b_g, expand=1)
    assert lib.switch_moe_sync_status() == 0
    for f in a._fields:
        assert torch.equal(getattr(a, f), getattr(b, f)), f


@pytest.mark.parametrize("kw,code", [
    (dict(expand=5), "INVALID_ARG"), (dict(expand=-1), "INVALID_ARG"),
    (dict(expand=2, priority_mode=1), "UNSUPPORTED"), (dict(expand=3, N=2), "UNSUPPORTED"),
])
def test_expand_argument_checks(kw, code):
    from switch_top_expert_router_b300 import build
    build.build()
    import switch_top_expert_router_b300 as sm
    args = dict(T=1000, d_model=64, d_ff=128, N=8, capacity_factor=1.0, priority_mode=0,
                gate_multiply=1, dtype=1, has_shared=0)
    args.update(kw)
    with pytest.raises(sm.SwitchMoEError) as ei:
        sm.switch_moe_workspace_bytes(sm.make_params(**args))
    assert ei.value.code == getattr(sm, "SWITCH_MOE_ERR_" + code)


def test_expand_workspace_grows():
    from switch_top_expert_router_b300 import build
    build.build()
    import switch_top_expert_router_b300 as sm
    p1 = sm.make_params(1000, 64, 128, 8, 1.0)
    p3 = sm.make_params(1000, 64, 128, 8, 1.0, expand=3)
    assert sm.switch_moe_workspace_bytes(p3) > sm.switch_moe_workspace_bytes(p1)
