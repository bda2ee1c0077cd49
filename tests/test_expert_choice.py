"""Expert-choice routing on the CUDA path against the oracle ("Top-1 路由
(Top-1 Routing)", compassingai.com, routing-paradigm table: each expert
selects its top-K tokens; comparison table: a token may be taken by several
experts or by none).

The selection compares fp32 scores (expf softmax) where the oracle has fp64
ones, so a token whose score lies within the gate tolerance of an expert's
k-th best score may fall on either side.  Checked:
* every chosen gate equals the token's fp64 score within the gate tolerance;
* each expert's list holds k = min(C, T) distinct tokens in (score desc,
  token asc) order of the kernel's own fp32 scores;
* a token clearly above the k-th fp64 score is taken, one clearly below is
  not; where the scores at the boundary are exactly equal (integer logits)
  the lower token indices are taken, exactly as the oracle does;
* experts_per_token counts the lists; expert_counts / aux_loss are the
  router's top-1 statistics (bit-exact / 1e-5 relative);
* y end to end within max|dy| / rms <= 1e-2 against the oracle's FFN and
  merge applied to the kernel's own selection.
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
    if kind == "ints":
        return torch.randint(-2, 3, (T, N), generator=g).float()
    if kind == "equal":
        return torch.zeros(T, N)
    raise ValueError(kind)


def check_selection(chosen, gates, probs64, C, rtol):
    T, N = probs64.shape
    k = min(C, T)
    chosen = np.asarray(chosen)
    gates = np.asarray(gates, dtype=np.float64)
    assert chosen.shape == (N, C)
    assert np.all(chosen[:, k:] == -1) and np.all(gates[:, k:] == 0)
    ch, gt = chosen[:, :k], gates[:, :k]
    want, _ = oracle.expert_choice(probs64, C)
    for e in range(N):
        toks = ch[e]
        assert len(set(toks.tolist())) == k and toks.min() >= 0 and toks.max() < T
        col = probs64[:, e]
        np.testing.assert_allclose(gt[e], col[toks], rtol=rtol, atol=0)
        # (gate desc, token asc) order of the kernel's own scores
        for i in range(k - 1):
            assert gt[e, i] > gt[e, i + 1] or (gt[e, i] == gt[e, i + 1] and toks[i] < toks[i + 1])
        s_k = np.sort(col)[::-1][k - 1]
        band = np.abs(col - s_k) <= rtol * s_k
        if np.all(col[band] == s_k):   # only exact ties at the boundary: decided by index
            assert sorted(toks.tolist()) == sorted(want[e].tolist()), f"expert {e}"
        else:
            taken = np.zeros(T, dtype=bool)
            taken[toks] = True
            assert np.all(taken[col > s_k * (1 + rtol)]), f"expert {e}: a clear winner left out"
            assert not np.any(taken[col < s_k * (1 - rtol)]), f"expert {e}: a clear loser taken"


ROUTE_CASES = [
    # T, N, cf, kind
    (8192, 128, 1.25, "normal"),
    (4096, 64, 2.0, "normal"),
    (1000, 7, 0.5, "ints"),         # exact ties at the boundaries
    (300, 4, 1.0, "equal"),         # every score equal: the first C tokens
    (50, 8, 16.0, "normal"),        # C > T: every expert takes every token
    (2048, 256, 0.75, "normal"),
    (20000, 8, 0.5, "normal"),      # radix select over 20000 keys, C = 1250
]


@pytest.mark.gpu
@pytest.mark.parametrize("T,N,cf,kind", ROUTE_CASES)
def test_route_expert_choice_matches_oracle(lib, T, N, cf, kind):
    logits = _logits(T, N, T * 7 + N, kind)
    gpu = lib.switch_moe_route_expert_choice(logits.cuda(), cf)
    assert lib.switch_moe_sync_status() == 0
    C = oracle.capacity(T, N, cf)
    ref = oracle.route_from_logits(logits)
    check_selection(np_(gpu.chosen_token), np_(gpu.chosen_gate), ref["probs"], C, GATE_RTOL)
    ch = np_(gpu.chosen_token)
    per = np.bincount(ch[ch >= 0], minlength=T)
    assert np.array_equal(np_(gpu.experts_per_token), per)
    assert np.array_equal(np_(gpu.expert_counts), np.bincount(ref["expert_id"], minlength=N))
    aux = oracle.aux_loss(ref["probs"], np.bincount(ref["expert_id"], minlength=N))
    assert abs(float(np_(gpu.aux_loss)[0]) - aux) <= AUX_TOL * abs(aux)


FWD_CASES = [
    # name, T, d, F, N, cf, dtype, gate_multiply, shared
    ("bf16-ffn", 4096, 256, 512, 32, 1.0, "bf16", 1, 0),
    ("bf16-ffn-cf2", 2048, 256, 512, 16, 2.0, "bf16", 1, 0),
    ("bf16-N200-tmem-router", 2048, 128, 256, 200, 1.5, "bf16", 1, 0),
    ("bf16-shared", 1000, 128, 256, 8, 1.2, "bf16", 1, 1),
    ("bf16-no-gate", 1000, 128, 256, 8, 1.0, "bf16", 0, 0),
    ("f32", 512, 64, 256, 8, 1.0, "f32", 1, 0),
    ("f32-shared", 300, 64, 128, 4, 1.5, "f32", 1, 1),
    ("bf16-big-C", 3000, 128, 256, 4, 1.2, "bf16", 1, 0),          # token tiles of 256
    ("bf16-decode", 64, 512, 1024, 8, 1.0, "bf16", 1, 0),         # 16-token tiles
    ("bf16-ksplit", 300, 512, 1024, 2, 1.0, "bf16", 1, 0),        # C = 150: K-split GEMM 2
    ("bf16-C-over-T", 40, 64, 128, 8, 16.0, "bf16", 1, 0),        # every expert takes all
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", FWD_CASES, ids=[c[0] for c in FWD_CASES])
def test_forward_expert_choice(lib, case):
    name, T, d, F, N, cf, dt, gm, sh = case
    w = Workload(name, T, d, F, N, cf, dt, 0.3, has_shared=sh)
    inp = make_inputs(w, seed=19, device="cuda")
    out = lib.switch_moe_forward_expert_choice(inp.x, inp.W_g, inp.W1, inp.W2, cf,
                                               gate_multiply=gm, b_g=inp.b_g, W1s=inp.W1s,
                                               W2s=inp.W2s)
    lg = lib.switch_moe_router_logits(inp.x, inp.W_g, inp.b_g)   # what the forward routed on
    assert lib.switch_moe_sync_status() == 0
    C = oracle.capacity(T, N, cf)
    ref = oracle.route_from_logits(lg.cpu())
    check_selection(np_(out.chosen_token), np_(out.chosen_gate), ref["probs"], C, GATE_RTOL)
    ch = np_(out.chosen_token)
    assert np.array_equal(np_(out.experts_per_token), np.bincount(ch[ch >= 0], minlength=T))
    assert np.array_equal(np_(out.expert_counts), np.bincount(ref["expert_id"], minlength=N))
    k = min(C, T)
    g64 = np.stack([ref["probs"][ch[e, :k], e] for e in range(N)])
    getter = lambda i: (inp.W1[i].cpu(), inp.W2[i].cpu())  # noqa: E731
    y_ref = oracle.forward_rows_expert_choice(np.arange(T), inp.x.cpu(), ch[:, :k], g64, gm,
                                              getter,
                                              None if inp.W1s is None else inp.W1s.cpu(),
                                              None if inp.W2s is None else inp.W2s.cpu())
    rms = np.sqrt((y_ref ** 2).mean())
    err = np.abs(np_(out.y).astype(np.float64) - y_ref).max() / rms
    assert err <= Y_TOL, f"y max|err|/rms = {err:.3g}"


@pytest.mark.gpu
def test_forward_expert_choice_oracle_end_to_end(lib):
    """A small layer run whole through the oracle's expert-choice forward."""
    w = Workload("e2e", 256, 64, 128, 8, 1.0, "bf16", 0.3)
    inp = make_inputs(w, seed=29, device="cuda")
    out = lib.switch_moe_forward_expert_choice(inp.x, inp.W_g, inp.W1, inp.W2, 1.0)
    assert lib.switch_moe_sync_status() == 0
    ref = oracle.forward_expert_choice(inp.x.cpu(), inp.W_g.cpu(), inp.W1.cpu(), inp.W2.cpu(),
                                       1.0)
    # no score of the seeded inputs sits within 1e-5 of an expert's boundary
    p = ref["probs"]
    k = ref["chosen"].shape[1]
    for e in range(8):
        srt = np.sort(p[:, e])[::-1]
        assert srt[k - 1] - srt[k] > 1e-5 * srt[k - 1]
    assert np.array_equal(np.sort(np_(out.chosen_token), axis=1), np.sort(ref["chosen"], axis=1))
    rms = np.sqrt((ref["y"] ** 2).mean())
    assert np.abs(np_(out.y).astype(np.float64) - ref["y"]).max() / rms <= Y_TOL


@pytest.mark.parametrize("kw,code", [
    (dict(expert_choice=2), "INVALID_ARG"),
    (dict(expert_choice=1, top_k=2), "UNSUPPORTED"),
    (dict(expert_choice=1, expand=2), "UNSUPPORTED"),
    (dict(expert_choice=1, T=40000, N=2, capacity_factor=1.0), "UNSUPPORTED"),   # C > 16384
])
def test_expert_choice_argument_checks(kw, code):
    from switch_top_expert_router_b300 import build
    build.build()
    import switch_top_expert_router_b300 as sm
    args = dict(T=1000, d_model=64, d_ff=128, N=8, capacity_factor=1.0, priority_mode=0,
                gate_multiply=1, dtype=1, has_shared=0)
    args.update(kw)
    with pytest.raises(sm.SwitchMoEError) as ei:
        sm.switch_moe_workspace_bytes(sm.make_params(**args))
    assert ei.value.code == getattr(sm, "SWITCH_MOE_ERR_" + code)


def test_expert_choice_workspace_holds_the_scores():
    from switch_top_expert_router_b300 import build
    build.build()
    import switch_top_expert_router_b300 as sm
    T, N = 8192, 128
    a = sm.switch_moe_workspace_bytes(sm.make_params(T, 768, 3072, N, 1.25))
    b = sm.switch_moe_workspace_bytes(sm.make_params(T, 768, 3072, N, 1.25, expert_choice=1))
    assert b - a >= T * N * 4    # the transposed probabilities
