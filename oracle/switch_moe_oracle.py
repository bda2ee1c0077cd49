"""Plain fp64 CPU oracle of the Switch top-1 MoE layer forward.

TEST INFRASTRUCTURE.  Only tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code,
header, table or helper with the CUDA library and never calls it.

Every step is the plain definition from the pages, one step after another,
in float64 (inputs are the exact bf16 / fp32 values widened to float64).
A library primitive (matmul, argmax, exp) serves as a step; there is no
blocking, fusion or reordering beyond the definitions.

Sources (page title, then section / equation / figure):

* [TOP1]  "Top-1 路由 (Top-1 Routing)", compassingai.com -- core mechanism
  steps 1-3 (gating softmax, top-1 argmax and gate value, expert output),
  load-balancing section (auxiliary loss), Token Dropping section
  (capacity per expert), key-parameter section (two-layer FFN, no bias).
* [SWITCH] Switch Transformer walk-through, personwebsite.pages.dev/moe-switch
  -- Switch layer (gate value as the multiplier, Eq. 2), expert capacity
  (dropped tokens skip the expert and ride the residual), load-balancing
  loss (Eq. 4, whose symbols f_i and P_i survive in the text), selective
  float32 router precision.
* [CAP]   "MoE 专家容量因子与 Token 丢弃", wiblog.cn -- capacity formula
  (section on where capacity comes from), overflow handling (section on
  what happens after overflow: sort by routing weight, keep the highest),
  the token-path flowchart (nodes D -> F: the capacity decision is taken
  after all scores are known and before any expert runs).
* [CMP]   "Which Routing Does Each MoE Model Use?" (MarkTechPost digest) --
  routing table: Llama 4 Maverick routes top-1 over 128 experts plus one
  always-on shared expert.

Readings where the pages are silent or disagree (each is a choice, made
once, and stated here):

* capacity rounds up: C = ceil(cf * T / N), evaluated in double as
  (cf * T) / N; C must be >= 1.
* argmax is taken on the logits (same order as on the softmax scores), and
  the lowest expert index wins exact ties.
* f_i counts the router's choices before capacity (tokens *routed* to i).
* gate-value priority orders an expert's tokens by (gate desc, token asc);
  the slot of a kept token is its rank in that order.  Token-order priority
  gives slot = number of earlier tokens with the same expert.
* a dropped token's MoE output is the zero vector; the caller adds the
  residual.  The shared expert (when present) runs on every token,
  dropped or not.
* the expert FFN is ReLU between two bias-free linear maps.
* whether the gate scales the expert output is a flag (TOP1 says Switch
  does not scale; SWITCH Eq. 2 says the gate is the multiplier).
"""
from __future__ import annotations

import math
from typing import Callable, Optional, Sequence

import numpy as np

__all__ = [
    "TOKEN_ORDER", "GATE_PRIORITY",
    "capacity", "router_logits", "softmax", "top1", "route", "route_from_logits",
    "assign_slots", "expert_ffn", "aux_loss", "combine_token", "forward",
    "forward_rows", "candidates", "assign_slots_expanded", "top2_gates",
    "assign_slots_top2", "forward_top2", "forward_rows_top2", "expert_choice",
    "forward_expert_choice", "forward_rows_expert_choice", "backward",
]

TOKEN_ORDER = 0
GATE_PRIORITY = 1


def _f64(a) -> np.ndarray:
    """Widen a numpy array or a (CPU) torch tensor of any float dtype to float64."""
    if hasattr(a, "detach"):  # torch tensor; bf16 has no numpy dtype
        a = a.detach().to("cpu")
        import torch  # local: numpy-only callers never need torch
        a = a.to(torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# Step a3: expert capacity.
#   [TOP1] Token Dropping section; [CAP] section on where capacity comes
#   from: capacity = capacity_factor * tokens_per_batch / num_experts.
#   Rounding is not on the pages: ceil, in double, in this evaluation order.
# --------------------------------------------------------------------------
def capacity(T: int, N: int, capacity_factor: float) -> int:
    if T <= 0 or N <= 0 or not (capacity_factor > 0) or math.isinf(capacity_factor):
        raise ValueError("capacity needs T > 0, N > 0 and a finite cf > 0")
    c = math.ceil(float(capacity_factor) * float(T) / float(N))
    if c < 1:
        raise ValueError("capacity rounds to zero")
    return int(c)


# --------------------------------------------------------------------------
# Step a1: router logits h = W_g . x  ([TOP1] core mechanism step 1,
# W_g in R^{N x d}; [SWITCH] router variable producing logits).  The
# optional per-expert bias b_g only serves to skew a synthetic workload.
# --------------------------------------------------------------------------
def router_logits(x, W_g, b_g=None) -> np.ndarray:
    x64 = _f64(x)
    W64 = _f64(W_g)
    logits = x64 @ W64.T                      # [T, N]
    if b_g is not None:
        logits = logits + _f64(b_g)[None, :]
    return logits


# Step a2: score = softmax(logits) over the N experts ([TOP1] step 1).
def softmax(logits) -> np.ndarray:
    l = _f64(logits)
    m = l.max(axis=1, keepdims=True)
    ex = np.exp(l - m)
    return ex / ex.sum(axis=1, keepdims=True)


# Step a2: expert_id = argmax(score), gate_value = score[expert_id]
# ([TOP1] step 2).  Argmax on the logits; the lowest index wins ties.
def top1(logits, probs):
    l = _f64(logits)
    p = _f64(probs)
    T = l.shape[0]
    expert_id = np.empty(T, dtype=np.int64)
    for t in range(T):
        row = l[t]
        best = 0
        for i in range(1, row.shape[0]):
            if row[i] > row[best]:           # strict: an equal later logit never wins
                best = i
        expert_id[t] = best
    gate = p[np.arange(T), expert_id]
    return expert_id, gate


def _top1_fast(l: np.ndarray, p: np.ndarray):
    # np.argmax returns the first maximal index, the same rule as top1();
    # used for large T where the per-token Python loop is too slow.
    e = np.argmax(l, axis=1).astype(np.int64)
    return e, p[np.arange(l.shape[0]), e]


def route(x, W_g, b_g=None):
    """Router of one batch: logits, probabilities, expert_id, gate (fp64)."""
    l = router_logits(x, W_g, b_g)
    p = softmax(l)
    e, g = (_top1_fast(l, p) if l.shape[0] > 4096 else top1(l, p))
    return {"logits": l, "probs": p, "expert_id": e, "gate": g}


def route_from_logits(logits32):
    """Routing decisions on given (fp32) logits; the comparisons that pick
    the expert see exactly those values (fp32 values are exact in fp64)."""
    l = _f64(logits32)
    p = softmax(l)
    e, g = (_top1_fast(l, p) if l.shape[0] > 4096 else top1(l, p))
    return {"logits": l, "probs": p, "expert_id": e, "gate": g}


# --------------------------------------------------------------------------
# Steps a4 / a4': slot assignment and overflow.
#   [SWITCH] expert capacity: tokens beyond an expert's capacity are dropped.
#   [CAP] overflow section + flowchart D -> F: sort an expert's tokens by
#   routing weight, keep the highest-weight ones, mark the rest overflow;
#   decided after all scores are known, before any expert computes.
# --------------------------------------------------------------------------
def assign_slots(expert_id, gate, N: int, C: int, priority_mode: int = TOKEN_ORDER):
    """Returns (slot int64[T] with -1 for dropped, drop uint8[T],
    counts int64[N] = tokens routed to each expert before capacity)."""
    e = np.asarray(expert_id, dtype=np.int64)
    T = e.shape[0]
    slot = np.full(T, -1, dtype=np.int64)
    counts = np.zeros(N, dtype=np.int64)
    if priority_mode == TOKEN_ORDER:
        for t in range(T):                    # a stable pass in token order
            pos = counts[e[t]]
            counts[e[t]] += 1
            if pos < C:
                slot[t] = pos
    elif priority_mode == GATE_PRIORITY:
        g = np.asarray(gate, dtype=np.float64)
        members = [[] for _ in range(N)]
        for t in range(T):
            members[e[t]].append(t)
        for i in range(N):
            counts[i] = len(members[i])
            order = sorted(members[i], key=lambda t: (-g[t], t))
            for rank, t in enumerate(order):
                if rank < C:
                    slot[t] = rank
    else:
        raise ValueError("priority_mode must be 0 (token order) or 1 (gate priority)")
    drop = (slot < 0).astype(np.uint8)
    return slot, drop, counts


# --------------------------------------------------------------------------
# Expanded Drop ([CAP] inference section, on Capacity-Aware Inference: the
# tokens an over-full expert drops consider further experts of their
# candidate set, so the spare capacity of under-used experts is used).
# The page gives the idea in one sentence; the reading taken here:
#   * a token's candidate set is its experts in descending logit order
#     (lowest index first on ties), the first k of them;
#   * pass 1 is the top-1 assignment with capacity C in token order;
#   * in pass r = 2..k every token still unplaced, in token order, takes
#     the next free slot of its r-th candidate if that expert has one;
#   * a token placed in pass r is processed by that expert, with that
#     expert's probability as its gate; expert_counts (f_i) and L_aux keep
#     the router's top-1 choices.
# k = 1 is the plain top-1 assignment.
# --------------------------------------------------------------------------
def candidates(logits, k: int) -> np.ndarray:
    """int64 [T, k]: each token's experts by descending logit, lowest index
    first among equal logits."""
    l = _f64(logits)
    order = np.argsort(-l, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def assign_slots_expanded(cands, N: int, C: int):
    """Returns (expert int64[T] processing each token -- its first
    candidate when dropped --, slot int64[T] with -1 for dropped,
    drop uint8[T], used int64[N] = filled slots per expert)."""
    cands = np.asarray(cands, dtype=np.int64)
    T, k = cands.shape
    used = np.zeros(N, dtype=np.int64)
    expert = cands[:, 0].copy()
    slot = np.full(T, -1, dtype=np.int64)
    for r in range(k):                        # pass r + 1
        for t in range(T):                    # token order
            if slot[t] >= 0:
                continue
            e = cands[t, r]
            if used[e] < C:
                slot[t] = used[e]
                used[e] += 1
                expert[t] = e
    drop = (slot < 0).astype(np.uint8)
    return expert, slot, drop, used


# --------------------------------------------------------------------------
# Top-2 token choice, the variant the pages set beside Switch's top-1:
#   [TOP1] industry-position and comparison sections (GShard, Mixtral:
#   every token goes to 2 experts, is sent twice and needs a weighted
#   merge); [SWITCH] Switch-layer section (Shazeer's top-k layer: logits
#   h = W_r x, softmax-normalised gate values, the output is the gate-weighted
#   sum over the chosen index set T); [CMP] routing table (Mixtral 8x7B:
#   softmax over the top-k).
# Readings, none of them printed on the pages:
#   * the chosen set is the 2 highest logits, lowest index first on ties
#     (candidates(logits, 2)); choice 0 is the top-1 expert;
#   * capacity keeps the printed formula C = ceil(cf * T / N) (a caller who
#     wants room for both choices passes a larger cf);
#   * slots: first every token's choice 0 in token order (the top-1
#     assignment), then every token's choice 1 in token order, after the
#     choices the expert already kept; a (token, choice) pair is kept iff
#     its slot < C;
#   * gates: the chosen experts' softmax probabilities, or with renormalize
#     the softmax over the two chosen logits, p_e / (p_e0 + p_e1);
#   * y_t = sum over the token's kept choices of gate * E(x_t); a dropped
#     choice adds nothing and the other gate is not re-scaled;
#   * expert_counts (f_i of L_aux) count choice 0, the router's top-1.
# --------------------------------------------------------------------------
def top2_gates(probs, cands, renormalize: int) -> np.ndarray:
    """float64 [T, 2]: the gate of each chosen expert."""
    p = _f64(probs)
    cands = np.asarray(cands, dtype=np.int64)
    rows = np.arange(p.shape[0])
    g = np.stack([p[rows, cands[:, 0]], p[rows, cands[:, 1]]], axis=1)
    if renormalize:
        g = g / g.sum(axis=1, keepdims=True)
    return g


def assign_slots_top2(cands, N: int, C: int):
    """Returns (slot int64[T, 2] with -1 for a dropped choice, drop uint8[T, 2],
    used int64[N] = filled slots per expert)."""
    cands = np.asarray(cands, dtype=np.int64)
    T = cands.shape[0]
    used = np.zeros(N, dtype=np.int64)
    slot = np.full((T, 2), -1, dtype=np.int64)
    for r in range(2):                        # all first choices, then all second
        for t in range(T):                    # token order
            e = cands[t, r]
            if used[e] < C:
                slot[t, r] = used[e]
                used[e] += 1
    return slot, (slot < 0).astype(np.uint8), used


# --------------------------------------------------------------------------
# Expert choice, the paradigm the pages set against token choice:
#   [TOP1] routing-paradigm table (each expert selects its top-K tokens,
#   balanced by construction), milestone table (Expert Choice Routing,
#   Zhou et al. 2022: the choice flips from tokens to experts) and the
#   comparison table (a token can be taken by several experts, or by none).
# Readings, none of them printed on the pages:
#   * the scores are the router of the top-1 layer: s[t, e] = softmax over
#     the N experts of token t's logits;
#   * each expert takes k = C = ceil(cf * T / N) tokens (all T when C >= T):
#     the highest s[:, e], the lower token index first among equal scores;
#     slot = rank in that order;
#   * y_t = sum over the experts that took t of s[t, e] * E_e(x_t) (the gate
#     flag as for top-1); a token no expert took gets 0 (plus the shared
#     expert);
#   * expert_counts and L_aux describe the router's top-1 choice, as for the
#     other variants (expert choice itself needs no balancing loss).
# --------------------------------------------------------------------------
def expert_choice(probs, C: int):
    """Returns (chosen int64 [N, min(C, T)]: each expert's tokens, best
    first; gates float64 [N, min(C, T)]: their scores)."""
    p = _f64(probs)
    T, N = p.shape
    k = min(C, T)
    chosen = np.zeros((N, k), dtype=np.int64)
    gates = np.zeros((N, k), dtype=np.float64)
    tok = np.arange(T)
    for e in range(N):
        order = np.lexsort((tok, -p[:, e]))   # score desc, then token asc
        chosen[e] = order[:k]
        gates[e] = p[order[:k], e]
    return chosen, gates


def forward_expert_choice(x, W_g, W1, W2, capacity_factor: float, gate_multiply: int = 1,
                          b_g=None, W1s=None, W2s=None,
                          expert_getter: Optional[Callable[[int], tuple]] = None):
    """The layer with expert-choice routing.  Returns a dict with y (fp64
    [T, d]), chosen / gates [N, min(C, T)], experts_per_token [T], counts
    of the router's top-1 choice and aux_loss."""
    r = route(x, W_g, b_g)
    T, N = r["probs"].shape
    C = capacity(T, N, capacity_factor)
    chosen, gates = expert_choice(r["probs"], C)
    d = x.shape[1]
    y = np.zeros((T, d), dtype=np.float64)
    for e in range(N):
        W1_e, W2_e = expert_getter(e) if expert_getter else (W1[e], W2[e])
        o = expert_ffn(_rows(x, chosen[e]), W1_e, W2_e)
        g = gates[e][:, None] if gate_multiply else 1.0
        np.add.at(y, chosen[e], g * o)          # one token may be taken by several experts
    if W1s is not None:
        y = y + expert_ffn(x, W1s, W2s)
    per_token = np.bincount(chosen.ravel(), minlength=T).astype(np.int64)
    counts = np.bincount(r["expert_id"], minlength=N).astype(np.int64)
    return {"y": y, "chosen": chosen, "gates": gates, "experts_per_token": per_token,
            "counts": counts, "aux_loss": aux_loss(r["probs"], counts),
            "logits": r["logits"], "probs": r["probs"], "capacity": C}


# --------------------------------------------------------------------------
# Step a6/a7: the expert, a two-layer bias-free FFN ([TOP1] key-parameter
# section: about 2 * d_model * d_ff weights per expert).  ReLU between.
#   W1_e: [d_ff, d_model], W2_e: [d_model, d_ff] (out-features first).
# --------------------------------------------------------------------------
def expert_ffn(x_rows, W1_e, W2_e) -> np.ndarray:
    xr = _f64(x_rows)
    h = xr @ _f64(W1_e).T                      # [n, d_ff]
    h = np.maximum(h, 0.0)
    return h @ _f64(W2_e).T                    # [n, d_model]


# --------------------------------------------------------------------------
# Step a10: L_aux = N * sum_i f_i * P_i  ([TOP1] load-balancing section;
# [SWITCH] Eq. 4 text): f_i = share of the batch's tokens routed to expert i,
# P_i = mean router probability of expert i over the batch.  Unscaled by
# the coefficient alpha (the caller applies it).
# --------------------------------------------------------------------------
def aux_loss(probs, counts) -> float:
    p = _f64(probs)
    T, N = p.shape
    f = np.asarray(counts, dtype=np.float64) / T
    P = p.sum(axis=0) / T
    return float(N * np.sum(f * P))


# Step a9: combine one token.  [TOP1] step 3 / [SWITCH] Eq. 2 (gate flag);
# [SWITCH] capacity section and [CAP] overflow section: a dropped token gets
# no expert output (zero vector; the residual is the caller's).
def combine_token(o_row: Optional[np.ndarray], gate: float, dropped: bool,
                  gate_multiply: bool, d_model: int,
                  shared_row: Optional[np.ndarray] = None) -> np.ndarray:
    if dropped:
        y = np.zeros(d_model, dtype=np.float64)
    else:
        y = (gate if gate_multiply else 1.0) * o_row
    if shared_row is not None:                 # [CMP]: shared expert is always on
        y = y + shared_row
    return y


def forward(x, W_g, W1, W2, capacity_factor: float, priority_mode: int = TOKEN_ORDER,
            gate_multiply: int = 1, b_g=None, W1s=None, W2s=None,
            expert_getter: Optional[Callable[[int], tuple]] = None, expand: int = 1):
    """The whole layer on one batch.

    W1 / W2 are [N, F, d] / [N, d, F]; alternatively ``expert_getter(e)``
    returns (W1_e, W2_e) so that large layers need not be held whole.
    expand > 1: Expanded Drop over the first `expand` candidates (token
    order only).  Returns a dict with y (fp64 [T, d]), routing outputs
    (expert_id / gate of the processing expert) and aux_loss."""
    r = route(x, W_g, b_g)
    T, N = r["probs"].shape
    C = capacity(T, N, capacity_factor)
    slot, drop, counts = assign_slots(r["expert_id"], r["gate"], N, C, priority_mode)
    expert_id, gate = r["expert_id"], r["gate"]
    if expand > 1:
        if priority_mode != TOKEN_ORDER:
            raise ValueError("Expanded Drop is defined for token-order priority")
        expert_id, slot, drop, _ = assign_slots_expanded(candidates(r["logits"], expand), N, C)
        gate = r["probs"][np.arange(T), expert_id]
    d = x.shape[1]
    y = np.zeros((T, d), dtype=np.float64)
    o = np.zeros((T, d), dtype=np.float64)
    for i in range(N):
        rows = np.nonzero((expert_id == i) & (slot >= 0))[0]
        if rows.size == 0:
            continue
        W1_e, W2_e = expert_getter(i) if expert_getter else (W1[i], W2[i])
        o[rows] = expert_ffn(_rows(x, rows), W1_e, W2_e)
    S = expert_ffn(x, W1s, W2s) if W1s is not None else None
    for t in range(T):
        y[t] = combine_token(o[t], gate[t], bool(drop[t]), bool(gate_multiply), d,
                             None if S is None else S[t])
    return {"y": y, "expert_id": expert_id, "gate": gate, "slot": slot,
            "drop": drop, "counts": counts, "aux_loss": aux_loss(r["probs"], counts),
            "logits": r["logits"], "probs": r["probs"], "capacity": C}


def forward_top2(x, W_g, W1, W2, capacity_factor: float, gate_multiply: int = 1,
                 renormalize: int = 0, b_g=None, W1s=None, W2s=None,
                 expert_getter: Optional[Callable[[int], tuple]] = None):
    """The layer with top-2 routing (token order).  Returns a dict with y
    (fp64 [T, d]), expert_id / gate / slot / drop as [T, 2] (choice 0 =
    the top-1 expert), counts of choice 0 and aux_loss."""
    r = route(x, W_g, b_g)
    T, N = r["probs"].shape
    if N < 2:
        raise ValueError("top-2 routing needs at least two experts")
    C = capacity(T, N, capacity_factor)
    cands = candidates(r["logits"], 2)
    gate = top2_gates(r["probs"], cands, renormalize)
    slot, drop, _ = assign_slots_top2(cands, N, C)
    counts = np.bincount(cands[:, 0], minlength=N).astype(np.int64)
    d = x.shape[1]
    o = np.zeros((T, 2, d), dtype=np.float64)
    for i in range(N):
        sel = [(t, c) for c in range(2) for t in np.nonzero((cands[:, c] == i) & (slot[:, c] >= 0))[0]]
        if not sel:
            continue
        W1_e, W2_e = expert_getter(i) if expert_getter else (W1[i], W2[i])
        ts = np.array([t for t, _ in sel])
        out = expert_ffn(_rows(x, ts), W1_e, W2_e)
        for k, (t, c) in enumerate(sel):
            o[t, c] = out[k]
    S = expert_ffn(x, W1s, W2s) if W1s is not None else None
    y = np.zeros((T, d), dtype=np.float64)
    for t in range(T):
        acc = np.zeros(d, dtype=np.float64)
        for c in range(2):                     # the weighted merge of the kept choices
            if not drop[t, c]:
                acc = acc + (gate[t, c] if gate_multiply else 1.0) * o[t, c]
        y[t] = acc if S is None else acc + S[t]
    return {"y": y, "expert_id": cands, "gate": gate, "slot": slot, "drop": drop,
            "counts": counts, "aux_loss": aux_loss(r["probs"], counts),
            "logits": r["logits"], "probs": r["probs"], "capacity": C}


# --------------------------------------------------------------------------
# Backward of the top-1 layer, for the training step the pages describe
# ([SWITCH] load-balancing section: the auxiliary loss is added to the
# training loss with a coefficient alpha; [TOP1] load-balancing section:
# L_aux = N * sum_i f_i P_i).  The loss seen here is <dy, y> + alpha * L_aux,
# so dy is the upstream gradient of y.  Readings:
#   * the routing decisions (argmax, capacity, slots) are piecewise constant
#     and get no gradient; f_i (argmax counts) is constant, so
#     dL_aux / dp[t, i] = N * f_i / T;
#   * the gate gets dy_t . E(x_t) when gate_multiply is set (y_t = g_t E(x_t));
#     a dropped token's expert branch is zero and passes no gradient;
#   * ReLU's derivative at 0 is taken as 0.
# Softmax backward: dl = p * (dp - sum_i p_i dp_i).
# --------------------------------------------------------------------------
def backward(x, W_g, W1, W2, capacity_factor: float, dy, priority_mode: int = TOKEN_ORDER,
             gate_multiply: int = 1, b_g=None, W1s=None, W2s=None, aux_coef: float = 0.0):
    """Gradients of <dy, y> + aux_coef * L_aux.  Returns a dict with dx,
    dW_g, db_g, dW1, dW2 (and dW1s, dW2s with a shared expert), all fp64."""
    fw = forward(x, W_g, W1, W2, capacity_factor, priority_mode, gate_multiply, b_g, W1s, W2s)
    x64, dy64 = _f64(x), _f64(dy)
    Wg64, W1_64, W2_64 = _f64(W_g), _f64(W1), _f64(W2)
    T, d = x64.shape
    N = Wg64.shape[0]
    e, g, slot = fw["expert_id"], fw["gate"], fw["slot"]
    dx = np.zeros_like(x64)
    dW1 = np.zeros_like(W1_64)
    dW2 = np.zeros_like(W2_64)
    dgate = np.zeros(T)
    for i in range(N):
        rows = np.nonzero((e == i) & (slot >= 0))[0]
        if rows.size == 0:
            continue
        xr = x64[rows]
        hpre = xr @ W1_64[i].T                   # [n, F]
        h = np.maximum(hpre, 0.0)
        o = h @ W2_64[i].T                       # [n, d]: E(x)
        scale = g[rows][:, None] if gate_multiply else 1.0
        dO = scale * dy64[rows]                  # through y = g * E(x)
        if gate_multiply:
            dgate[rows] = np.sum(dy64[rows] * o, axis=1)
        dW2[i] = dO.T @ h
        dh = (dO @ W2_64[i]) * (hpre > 0)
        dW1[i] = dh.T @ xr
        dx[rows] += dh @ W1_64[i]
    out = {"dW1": dW1, "dW2": dW2}
    if W1s is not None:
        W1s64, W2s64 = _f64(W1s), _f64(W2s)
        hpre = x64 @ W1s64.T
        h = np.maximum(hpre, 0.0)
        out["dW2s"] = dy64.T @ h
        dh = (dy64 @ W2s64) * (hpre > 0)
        out["dW1s"] = dh.T @ x64
        dx += dh @ W1s64
    p = fw["probs"]
    dp = np.zeros_like(p)
    dp[np.arange(T), e] += dgate                 # the gate is p[t, e_t]
    f = fw["counts"] / T
    dp += aux_coef * N * f[None, :] / T          # dL_aux / dp[t, i]
    dl = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
    out["dW_g"] = dl.T @ x64
    out["db_g"] = dl.sum(axis=0)
    dx += dl @ Wg64
    out["dx"] = dx
    out["forward"] = fw
    return out


def forward_rows(rows: Sequence[int], x, expert_id, gate, slot, gate_multiply: int,
                 expert_getter: Callable[[int], tuple], W1s=None, W2s=None) -> np.ndarray:
    """y for a sample of tokens, given routing decisions (for layers too large
    to run whole): rows are grouped by expert so each expert is fetched once."""
    rows = np.asarray(rows, dtype=np.int64)
    d = x.shape[1]
    out = np.zeros((rows.size, d), dtype=np.float64)
    e = np.asarray(expert_id)[rows]
    s = np.asarray(slot)[rows]
    g = np.asarray(gate, dtype=np.float64)[rows]
    xr = _rows(x, rows)
    o = np.zeros((rows.size, d), dtype=np.float64)
    for i in np.unique(e[s >= 0]):
        sel = np.nonzero((e == i) & (s >= 0))[0]
        W1_e, W2_e = expert_getter(int(i))
        o[sel] = expert_ffn(xr[sel], W1_e, W2_e)
    S = expert_ffn(xr, W1s, W2s) if W1s is not None else None
    for k in range(rows.size):
        out[k] = combine_token(o[k], g[k], bool(s[k] < 0), bool(gate_multiply), d,
                               None if S is None else S[k])
    return out


def forward_rows_top2(rows: Sequence[int], x, expert_id, gate, slot, gate_multiply: int,
                      expert_getter: Callable[[int], tuple], W1s=None, W2s=None) -> np.ndarray:
    """forward_rows under top-2 routing decisions (expert_id, gate, slot as
    [T, 2]): the sum of the two choices' rows, the shared expert once."""
    e, g, s = (np.asarray(a) for a in (expert_id, gate, slot))
    first = forward_rows(rows, x, e[:, 0], g[:, 0], s[:, 0], gate_multiply, expert_getter,
                         W1s, W2s)
    second = forward_rows(rows, x, e[:, 1], g[:, 1], s[:, 1], gate_multiply, expert_getter)
    return first + second


def forward_rows_expert_choice(rows: Sequence[int], x, chosen, gates, gate_multiply: int,
                               expert_getter: Callable[[int], tuple], W1s=None,
                               W2s=None) -> np.ndarray:
    """y for a sample of tokens under given expert-choice decisions
    (chosen / gates [N, k]): each sampled token's sum over the experts that
    took it."""
    rows = np.asarray(rows, dtype=np.int64)
    chosen = np.asarray(chosen)
    gates = np.asarray(gates, dtype=np.float64)
    d = x.shape[1]
    xr = _rows(x, rows)
    out = np.zeros((rows.size, d), dtype=np.float64)
    where = {int(t): k for k, t in enumerate(rows)}
    for e in range(chosen.shape[0]):
        hit = [(where[int(t)], g) for t, g in zip(chosen[e], gates[e]) if int(t) in where]
        if not hit:
            continue
        W1_e, W2_e = expert_getter(e)
        ks = np.array([k for k, _ in hit])
        o = expert_ffn(xr[ks], W1_e, W2_e)
        g = np.array([g for _, g in hit])[:, None] if gate_multiply else 1.0
        np.add.at(out, ks, g * o)
    if W1s is not None:
        out = out + expert_ffn(xr, W1s, W2s)
    return out


def _rows(x, rows):
    if hasattr(x, "detach"):
        import torch
        return _f64(x[torch.as_tensor(rows, dtype=torch.long, device=x.device)])
    return _f64(x)[rows]
