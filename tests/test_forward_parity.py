"""End-to-end parity of switch_moe_forward (CUDA) against the fp64 oracle.

Small layers: the oracle runs the whole batch.  Full-size layers (the four
bf16 shapes, in the launch configuration the benchmark times): the oracle
routes every token and computes y for a seeded sample of rows.
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import AUX_TOL, MARGIN, check_forward, near_tie_mask, np_
from workloads import CONFIGS, Workload, expert_weights, make_inputs, zipf_bias

pytestmark = pytest.mark.gpu


def run_gpu(lib, w: Workload, inp, ws=None):
    out = lib.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, w.capacity_factor,
                                 w.priority_mode, w.gate_multiply, b_g=inp.b_g,
                                 W1s=inp.W1s, W2s=inp.W2s, ws=ws)
    rc = lib.switch_moe_sync_status()
    assert rc == 0, lib.strerror(rc)
    return out


def oracle_full(w: Workload, inp):
    return oracle.forward(inp.x.cpu(), inp.W_g.cpu(), inp.W1.cpu(), inp.W2.cpu(),
                          w.capacity_factor, w.priority_mode, w.gate_multiply,
                          b_g=None if inp.b_g is None else inp.b_g.cpu(),
                          W1s=None if inp.W1s is None else inp.W1s.cpu(),
                          W2s=None if inp.W2s is None else inp.W2s.cpu())


SMALL = [
    # name, T, d, F, N, cf, dtype, mode, gm, shared
    ("tiny-layer", 512, 64, 256, 8, 1.0, "f32", 0, 1, 0),
    ("bf16-ragged", 777, 192, 320, 6, 1.25, "bf16", 0, 1, 0),     # F not a multiple of 128
    ("bf16-gate-prio", 1500, 128, 256, 16, 1.0, "bf16", 1, 1, 0),
    ("bf16-no-gate-mul", 600, 128, 256, 8, 1.0, "bf16", 0, 0, 0),
    ("bf16-shared", 300, 128, 384, 4, 1.0, "bf16", 0, 1, 1),
    ("bf16-multi-token-tiles", 3000, 128, 256, 4, 1.0, "bf16", 0, 1, 0),  # C = 750: 3 tiles
    ("bf16-decode", 64, 512, 1024, 8, 2.0, "bf16", 0, 1, 0),       # 16-token tiles, one launch
    ("bf16-ksplit", 300, 512, 1024, 2, 1.0, "bf16", 0, 1, 0),     # C = 150: K-split GEMM 2
    ("bf16-odd-d", 200, 72, 136, 3, 1.0, "bf16", 0, 1, 0),        # K and M tails (TMA zero fill)
    ("bf16-one-expert", 257, 128, 128, 1, 1.0, "bf16", 0, 1, 0),  # dense FFN
    ("bf16-one-token", 1, 64, 128, 4, 1.0, "bf16", 0, 1, 0),
    ("bf16-cf-ge-N", 400, 64, 128, 4, 4.0, "bf16", 1, 1, 0),      # nothing dropped
    ("bf16-C1", 400, 64, 128, 4, 0.01, "bf16", 0, 1, 0),          # C = 1
    ("f32-gate-prio-shared", 700, 96, 160, 5, 0.8, "f32", 1, 0, 1),
    ("bf16-big-C", 2000, 64, 256, 2, 1.0, "bf16", 1, 1, 1),       # C = 1000, gate prio, shared
    # 512 weight tiles per GEMM on a 148-CTA grid: the last 68 run as two K pieces each
    ("bf16-tail-split", 2048, 1024, 1024, 64, 1.0, "bf16", 0, 1, 0),
    ("bf16-tail-split-gate-shared", 2048, 1024, 1024, 64, 1.0, "bf16", 1, 0, 1),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_forward_small(lib, case):
    name, T, d, F, N, cf, dt, mode, gm, sh = case
    w = Workload(name, T, d, F, N, cf, dt, 0.3 if N > 1 else 0.1, priority_mode=mode,
                 gate_multiply=gm, has_shared=sh)
    inp = make_inputs(w, seed=7, device="cuda")
    out = run_gpu(lib, w, inp)
    ref = oracle_full(w, inp)
    info = check_forward(out, ref, N, ref["capacity"], mode)
    if N == 1:
        assert np.all(np_(out.gate) == 1.0)
    if cf >= N:
        assert info["dropped"] == 0


def test_zero_router_routes_everything_to_expert0(lib):
    w = Workload("zero-router", 300, 64, 128, 4, 1.0, "bf16", 0.0)
    inp = make_inputs(w, seed=1, device="cuda")
    inp.W_g.zero_()
    out = run_gpu(lib, w, inp)
    C = oracle.capacity(300, 4, 1.0)
    assert np.all(np_(out.expert_id) == 0)
    assert np.array_equal(np_(out.slot)[:C], np.arange(C)) and np.all(np_(out.slot)[C:] == -1)
    assert np.all(np_(out.y)[C:] == 0.0)
    assert float(np_(out.aux_loss)[0]) == pytest.approx(1.0, rel=AUX_TOL)
    ref = oracle_full(w, inp)
    rms = np.sqrt((ref["y"] ** 2).mean())
    assert np.abs(np_(out.y) - ref["y"]).max() / rms <= 1e-2


@pytest.mark.parametrize("name", ["base", "skew", "wide", "decode"])
def test_forward_full_size_sampled(lib, name):
    w = CONFIGS[name]
    inp = make_inputs(w, seed=0, device="cuda")
    out = run_gpu(lib, w, inp)
    # oracle: routing of every token, y of a seeded row sample
    r = oracle.route(inp.x.cpu(), inp.W_g.cpu(), None if inp.b_g is None else inp.b_g.cpu())
    C = oracle.capacity(w.T, w.N, w.capacity_factor)
    slot, drop, counts = oracle.assign_slots(r["expert_id"], r["gate"], w.N, C, w.priority_mode)
    ref = dict(r, slot=slot, drop=drop, counts=counts, aux_loss=oracle.aux_loss(r["probs"], counts))
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(w.T, size=min(w.T, 128 if name == "wide" else 384), replace=False))
    getter = lambda e: (inp.W1[e].cpu(), inp.W2[e].cpu())  # noqa: E731
    y_rows = oracle.forward_rows(rows, inp.x, r["expert_id"], r["gate"], slot, w.gate_multiply,
                                 getter,
                                 None if inp.W1s is None else inp.W1s.cpu(),
                                 None if inp.W2s is None else inp.W2s.cpu())
    info = check_forward(out, ref, w.N, C, w.priority_mode, rows, y_rows)
    print(f"{name}: near-ties={info['near_ties']} flips={info['flips']} "
          f"dropped={info['dropped']} y_err={info['y_err']:.2e}")
    if name == "skew":
        assert 0.10 <= info["dropped"] / w.T <= 0.30


def test_router_logits_and_route_consistency(lib):
    w = CONFIGS["base"]
    inp = make_inputs(w, seed=0, device="cuda", with_experts=False)
    lg = lib.switch_moe_router_logits(inp.x, inp.W_g)
    ref = oracle.router_logits(inp.x.cpu(), inp.W_g.cpu())
    scale = np.abs(ref).max()
    assert np.abs(np_(lg).astype(np.float64) - ref).max() <= 1e-6 * max(scale, 1.0) * 10
    # the logits the forward routes on are these, bit for bit
    W1 = torch.zeros((w.N, 16, w.d_model), dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros((w.N, w.d_model, 16), dtype=torch.bfloat16, device="cuda")
    fwd = lib.switch_moe_forward(inp.x, inp.W_g, W1, W2, w.capacity_factor)
    rt = lib.switch_moe_route_from_logits(lg, w.capacity_factor)
    assert lib.switch_moe_sync_status() == 0
    for k in ("expert_id", "gate", "slot", "drop_mask", "expert_counts", "aux_loss"):
        assert torch.equal(getattr(fwd, k), getattr(rt, k)), k
    assert np.all(np_(fwd.y) == 0.0)
    assert near_tie_mask(ref).sum() == 0   # the base shape has no margin below MARGIN
    assert MARGIN == 1e-5


def test_hostio_matches_device_path(lib):
    w = Workload("hostio", 1000, 128, 256, 8, 1.0, "bf16", 0.2, has_shared=1)
    inp = make_inputs(w, seed=3, device="cuda")
    dev = run_gpu(lib, w, inp)
    x_host = inp.x.cpu().pin_memory()
    host = lib.switch_moe_forward_hostio(x_host, inp.W_g, inp.W1, inp.W2, w.capacity_factor,
                                         W1s=inp.W1s, W2s=inp.W2s)
    torch.cuda.synchronize()
    for k in dev._fields:
        assert torch.equal(getattr(dev, k).cpu(), getattr(host, k)), k


def test_forward_deterministic_and_workspace_reuse(lib):
    w = Workload("det", 2048, 256, 512, 16, 1.0, "bf16", 0.2)
    inp = make_inputs(w, seed=5, device="cuda")
    ws = torch.full((lib.switch_moe_workspace_bytes(lib.make_params(2048, 256, 512, 16, 1.0)),),
                    255, dtype=torch.uint8, device="cuda")   # garbage on entry must not matter
    a = run_gpu(lib, w, inp, ws)
    b = run_gpu(lib, w, inp, ws)
    for k in a._fields:
        assert torch.equal(getattr(a, k), getattr(b, k)), k


def test_empty_batch_forward(lib):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    W_g = torch.zeros((4, 64), device="cuda")
    W1 = torch.zeros((4, 128, 64), dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros((4, 64, 128), dtype=torch.bfloat16, device="cuda")
    o = lib.switch_moe_forward(x, W_g, W1, W2, 1.0)
    assert lib.switch_moe_sync_status() == 0
    assert np.all(np_(o.expert_counts) == 0) and float(np_(o.aux_loss)[0]) == 0.0
