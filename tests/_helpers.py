"""Comparison helpers for the GPU parity tests (CUDA path vs CPU oracle)."""
import numpy as np
import torch

import oracle

# Tolerances of the parity contract:
#   routing/capacity/drop outputs: bit-exact (integers) when both sides see
#     the same fp32 logits; end to end, tokens whose fp64 top-1/top-2 logit
#     margin is below MARGIN are counted and excluded from the expert_id check
#   y: max|dy| / rms(y_ref) <= Y_TOL (bf16 operands, fp32 accumulation)
#   aux_loss: relative AUX_TOL
MARGIN = 1e-5
Y_TOL = 1e-2
AUX_TOL = 1e-5
GATE_RTOL = 2e-6      # fp32 softmax with expf vs fp64, on identical logits
U32 = 2.0 ** -24


def gate_rtol_e2e(logits64: np.ndarray, d: int) -> float:
    """Relative gate tolerance end to end, where the kernel's logits are fp32
    dot products of length d.  Summing d products in fp32 leaves a rounding
    error whose standard deviation is about u * rms(logit) * sqrt(d / 6)
    (u = 2^-24; the partial sums grow like sqrt(k)); the gate moves by the
    difference of two such errors.  20 standard deviations, and never less
    than the softmax's own rounding."""
    sigma = U32 * float(np.sqrt((logits64 ** 2).mean())) * np.sqrt(d / 6.0)
    return max(GATE_RTOL, 20.0 * sigma)


def np_(t):
    return t.detach().cpu().numpy()


def near_tie_mask(logits64: np.ndarray) -> np.ndarray:
    top2 = np.sort(logits64, axis=1)[:, -2:] if logits64.shape[1] > 1 else None
    if top2 is None:
        return np.zeros(logits64.shape[0], dtype=bool)
    return (top2[:, 1] - top2[:, 0]) < MARGIN


def gate_tie_experts(expert_id, gate, N, rtol=GATE_RTOL):
    """Experts holding two tokens whose gates differ by less than rtol (so
    fp32 and fp64 may order them differently in gate-priority mode)."""
    out = set()
    for i in range(N):
        g = np.sort(np.asarray(gate, dtype=np.float64)[np.asarray(expert_id) == i])
        if g.size > 1 and np.any(np.diff(g) <= rtol * g[1:]):
            out.add(i)
    return out


def check_routing_same_logits(gpu, logits32: torch.Tensor, N: int, C: int, mode: int):
    """GPU routing of given fp32 logits vs the oracle on the same logits."""
    ref = oracle.route_from_logits(logits32.cpu())
    e = np_(gpu.expert_id).astype(np.int64)
    assert np.array_equal(e, ref["expert_id"]), "expert_id differs on identical logits"
    g32 = np_(gpu.gate)
    np.testing.assert_allclose(g32.astype(np.float64), ref["gate"], rtol=GATE_RTOL, atol=0)
    # slot/drop/counts: the priority decision taken on the fp32 gates the
    # kernel decided with (same precision on both sides) -- bit-exact
    slot, drop, counts = oracle.assign_slots(e, g32, N, C, mode)
    assert np.array_equal(np_(gpu.slot), slot)
    assert np.array_equal(np_(gpu.drop_mask), drop)
    assert np.array_equal(np_(gpu.expert_counts), counts)
    # independent: the oracle's own fp64 gates; only experts with a gate
    # near-tie may differ, and only in gate-priority mode
    slot2, _, _ = oracle.assign_slots(ref["expert_id"], ref["gate"], N, C, mode)
    bad = set(np.unique(ref["expert_id"][slot2 != np_(gpu.slot)]).tolist())
    excused = gate_tie_experts(ref["expert_id"], ref["gate"], N) if mode == 1 else set()
    assert bad <= excused, f"slot mismatch in experts {sorted(bad - excused)}"
    aux_ref = oracle.aux_loss(ref["probs"], ref_counts := counts)
    assert abs(float(np_(gpu.aux_loss)[0]) - aux_ref) <= AUX_TOL * abs(aux_ref)
    return {"excused_experts": len(excused & bad), "counts": ref_counts}


def check_forward(out, ref, N, C, mode, y_rows=None, y_ref_rows=None):
    """GPU forward vs an oracle run of the same inputs.

    ref: oracle routing of the whole batch (dict with logits, expert_id,
    gate, slot, drop, counts, probs, aux_loss) and, unless y_rows is given,
    y for every token.  y_rows/y_ref_rows: a sample of token rows and the
    oracle's y for them."""
    e = np_(out.expert_id).astype(np.int64)
    near = near_tie_mask(ref["logits"])
    agree = e == ref["expert_id"]
    assert np.all(agree | near), f"{int((~agree & ~near).sum())} tokens routed differently"
    n_flip = int((~agree).sum())
    g32 = np_(out.gate)
    ok = agree
    d = np_(out.y).shape[1]
    np.testing.assert_allclose(g32[ok].astype(np.float64), ref["gate"][ok],
                               rtol=gate_rtol_e2e(ref["logits"], d))
    # validity: slots are exactly what the definition gives for the GPU's own
    # decisions (bit-exact)
    slot, drop, counts = oracle.assign_slots(e, g32, N, C, mode)
    assert np.array_equal(np_(out.slot), slot)
    assert np.array_equal(np_(out.drop_mask), drop)
    assert np.array_equal(np_(out.expert_counts), counts)
    # independent: against the oracle's own routing, outside experts touched
    # by a near-tie flip (and gate near-ties in gate-priority mode)
    touched = set(e[~agree].tolist()) | set(ref["expert_id"][~agree].tolist())
    if mode == 1:
        touched |= gate_tie_experts(ref["expert_id"], ref["gate"], N,
                                    gate_rtol_e2e(ref["logits"], d))
    clean = ~np.isin(ref["expert_id"], list(touched)) & ~np.isin(e, list(touched))
    assert np.array_equal(np_(out.slot)[clean], ref["slot"][clean])
    if not touched:
        assert np.array_equal(np_(out.expert_counts), ref["counts"])
    # y: tokens whose expert and keep status agree
    same = clean & (np_(out.drop_mask) == ref["drop"])
    y = np_(out.y).astype(np.float64)
    if y_rows is None:
        y_ref = ref["y"]
        rms = np.sqrt((y_ref ** 2).mean())
        err = np.abs(y[same] - y_ref[same]).max() / rms if same.any() else 0.0
    else:
        rows = np.asarray(y_rows)
        keep = same[rows]
        rms = np.sqrt((y_ref_rows ** 2).mean())
        err = np.abs(y[rows][keep] - y_ref_rows[keep]).max() / rms if keep.any() else 0.0
    assert err <= Y_TOL, f"y max|err|/rms = {err:.3g}"
    aux = float(np_(out.aux_loss)[0])
    assert abs(aux - ref["aux_loss"]) <= AUX_TOL * abs(ref["aux_loss"]), (aux, ref["aux_loss"])
    return {"near_ties": int(near.sum()), "flips": n_flip, "y_err": float(err),
            "dropped": int(np_(out.drop_mask).sum())}
