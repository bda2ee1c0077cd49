"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than itself: a value
worked by hand from the pages' formulas (tests/golden/), a closed form, a
brute-force definition on tiny inputs, an invariant, or a library routine
that computes the same special case.  They run without a GPU.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from oracle import switch_moe_oracle as OM

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- capacity
def _golden_capacity():
    rows = []
    with open(os.path.join(GOLDEN, "capacity.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                T, N, cf, C = line.split()
                rows.append((int(T), int(N), float(cf), int(C)))
    return rows


@pytest.mark.parametrize("T,N,cf,C", _golden_capacity())
def test_capacity_golden(T, N, cf, C):
    assert O.capacity(T, N, cf) == C


def test_capacity_properties():
    rng = np.random.default_rng(0)
    for _ in range(2000):
        T = int(rng.integers(1, 100000))
        N = int(rng.integers(1, 512))
        cf = float(rng.uniform(0.05, 4.0))
        C = O.capacity(T, N, cf)
        # C is the least integer with C >= cf*T/N (checked in exact rationals
        # for the double value of cf)
        from fractions import Fraction
        exact = Fraction(cf) * T / N
        assert C >= exact or math.isclose(C, float(exact), rel_tol=0, abs_tol=1e-9)
        assert C - 1 < exact + Fraction(1, 10**9)
        # cf >= N makes room for the whole batch in any one expert
        if cf >= N:
            assert C >= T
    for bad in [(0, 4, 1.0), (4, 0, 1.0), (4, 4, 0.0), (4, 4, -1.0), (4, 4, float("inf")),
                (4, 4, float("nan"))]:
        with pytest.raises(ValueError):
            O.capacity(*bad)


# ---------------------------------------------------------------- aux loss
def _golden_aux():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "aux_loss.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "case":
                cur = {"name": tok[1], "N": int(tok[3]), "expected": float(tok[5]), "p": []}
                cases.append(cur)
            elif tok[0] == "p":
                cur["p"].append([float(v) for v in tok[1:]])
    return cases


@pytest.mark.parametrize("case", _golden_aux(), ids=lambda c: c["name"])
def test_aux_loss_golden(case):
    p = np.array(case["p"], dtype=np.float64)
    assert p.shape[1] == case["N"]
    # routed expert = argmax of the probability row, lowest index on ties
    e, _ = O.top1(p, p)
    _, _, counts = O.assign_slots(e, p[np.arange(len(p)), e], case["N"], len(p))
    assert O.aux_loss(p, counts) == pytest.approx(case["expected"], rel=1e-14, abs=1e-14)


def test_aux_loss_zero_router_is_one():
    # W_g = 0: every logit equal, P_i = 1/N exactly, all tokens tie to expert 0
    for N in (1, 2, 7, 128):
        x = np.random.default_rng(N).standard_normal((37, 16))
        r = O.route(x, np.zeros((N, 16)))
        assert np.all(r["expert_id"] == 0)
        np.testing.assert_allclose(r["probs"], 1.0 / N, rtol=0, atol=1e-15)
        _, _, counts = O.assign_slots(r["expert_id"], r["gate"], N, 37)
        assert O.aux_loss(r["probs"], counts) == pytest.approx(1.0, abs=1e-14)


def test_aux_loss_balanced_routing_is_one():
    # token t -> expert t mod N (T a multiple of N) gives f_i = 1/N, so
    # L_aux = sum_i P_i = 1 whatever the probabilities are.
    rng = np.random.default_rng(1)
    N, T = 5, 40
    logits = rng.standard_normal((T, N))
    for t in range(T):
        logits[t, t % N] = logits[t].max() + 1.0
    r = O.route_from_logits(logits)
    assert np.array_equal(r["expert_id"], np.arange(T) % N)
    _, _, counts = O.assign_slots(r["expert_id"], r["gate"], N, T)
    assert O.aux_loss(r["probs"], counts) == pytest.approx(1.0, abs=1e-14)


def test_aux_loss_bounds():
    rng = np.random.default_rng(2)
    for _ in range(200):
        N = int(rng.integers(1, 9))
        T = int(rng.integers(1, 30))
        r = O.route_from_logits(rng.standard_normal((T, N)) * 3)
        _, _, counts = O.assign_slots(r["expert_id"], r["gate"], N, T)
        L = O.aux_loss(r["probs"], counts)
        assert 0.0 < L <= N + 1e-12


# ---------------------------------------------------------------- router
def test_router_logits_closed_form():
    # W_g rows = unit vectors e_{k_i}: logit i is coordinate k_i of x, plus bias
    rng = np.random.default_rng(3)
    x = rng.standard_normal((11, 9))
    ks = [4, 0, 8, 2]
    W = np.zeros((4, 9))
    for i, k in enumerate(ks):
        W[i, k] = 1.0
    b = np.array([0.5, -1.0, 0.0, 2.0])
    l = O.router_logits(x, W, b)
    assert l.shape == (11, 4)
    for i, k in enumerate(ks):
        np.testing.assert_array_equal(l[:, i], x[:, k] + b[i])


def test_router_logits_scaled_rows():
    # W_g = diag(s) restricted to the first N coordinates: logit i = s_i * x_i
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 5))
    s = np.array([2.0, -3.0, 0.5])
    W = np.zeros((3, 5))
    W[np.arange(3), np.arange(3)] = s
    np.testing.assert_allclose(O.router_logits(x, W), x[:, :3] * s, rtol=0, atol=0)


def test_softmax_against_torch():
    rng = np.random.default_rng(5)
    l = rng.standard_normal((50, 13)) * 4
    ref = torch.softmax(torch.from_numpy(l), dim=1).numpy()
    p = O.softmax(l)
    np.testing.assert_allclose(p, ref, rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    # shift invariance and overflow safety
    np.testing.assert_allclose(O.softmax(l + 700.0), p, rtol=1e-12, atol=1e-16)


def test_top1_ties_and_gate_closed_form():
    l = np.array([[0.0, 0.0, 0.0], [1.0, 3.0, 3.0], [2.0, -1.0, 2.0], [-5.0, -4.0, -4.5]])
    p = O.softmax(l)
    e, g = O.top1(l, p)
    assert list(e) == [0, 1, 0, 1]
    assert g[0] == pytest.approx(1 / 3, abs=1e-15)
    # two experts: gate = 1 / (1 + exp(-(a - b))) for the winner a
    rng = np.random.default_rng(6)
    ab = rng.standard_normal((100, 2)) * 2
    e, g = O.top1(ab, O.softmax(ab))
    margin = np.abs(ab[:, 0] - ab[:, 1])
    np.testing.assert_allclose(g, 1.0 / (1.0 + np.exp(-margin)), rtol=1e-14)
    assert np.all(e == np.where(ab[:, 1] > ab[:, 0], 1, 0))


def test_top1_fast_path_matches_loop():
    rng = np.random.default_rng(7)
    l = rng.integers(-2, 3, size=(300, 6)).astype(np.float64)  # many exact ties
    p = O.softmax(l)
    e1, g1 = O.top1(l, p)
    e2, g2 = OM._top1_fast(l, p)
    assert np.array_equal(e1, e2) and np.array_equal(g1, g2)
    big = rng.integers(-2, 3, size=(5000, 4)).astype(np.float64)
    r = O.route_from_logits(big)
    for t in range(0, 5000, 97):
        row = list(big[t])
        assert r["expert_id"][t] == row.index(max(row))


# ---------------------------------------------------------------- slots
def _brute(expert_id, gate, C, mode):
    """Definition: a token is kept iff fewer than C tokens of its expert come
    before it in priority order; its slot is that count."""
    T = len(expert_id)
    slot = np.full(T, -1)
    for t in range(T):
        ahead = 0
        for u in range(T):
            if u == t or expert_id[u] != expert_id[t]:
                continue
            if mode == O.TOKEN_ORDER:
                ahead += u < t
            else:
                ahead += (gate[u] > gate[t]) or (gate[u] == gate[t] and u < t)
        if ahead < C:
            slot[t] = ahead
    return slot


@pytest.mark.parametrize("mode", [O.TOKEN_ORDER, O.GATE_PRIORITY])
def test_assign_slots_bruteforce_all_assignments(mode):
    rng = np.random.default_rng(8)
    for N in (1, 2, 3):
        for T in range(1, 7 if N == 3 else 8):
            for assign in itertools.product(range(N), repeat=T):
                e = np.array(assign)
                gate = rng.permutation(T) / T + 0.01         # distinct gates
                if mode == O.GATE_PRIORITY and T >= 3 and rng.random() < 0.3:
                    gate[rng.integers(T)] = gate[rng.integers(T)]  # plant a tie
                for C in range(1, T + 1):
                    slot, drop, counts = O.assign_slots(e, gate, N, C, mode)
                    ref = _brute(e, gate, C, mode)
                    assert np.array_equal(slot, ref), (mode, N, T, assign, C)
                    assert np.array_equal(drop, (ref < 0).astype(np.uint8))
                    assert np.array_equal(counts, np.bincount(e, minlength=N))


@pytest.mark.parametrize("mode", [O.TOKEN_ORDER, O.GATE_PRIORITY])
def test_assign_slots_invariants(mode):
    rng = np.random.default_rng(9)
    for _ in range(50):
        N = int(rng.integers(1, 9))
        T = int(rng.integers(1, 400))
        C = int(rng.integers(1, T + 1))
        e = rng.integers(0, N, size=T)
        g = rng.random(T)
        slot, drop, counts = O.assign_slots(e, g, N, C, mode)
        assert counts.sum() == T
        for i in range(N):
            mine = np.nonzero(e == i)[0]
            kept = mine[slot[mine] >= 0]
            assert kept.size == min(counts[i], C)
            assert sorted(slot[kept]) == list(range(kept.size))     # a permutation
            dropped = mine[slot[mine] < 0]
            if mode == O.TOKEN_ORDER:
                assert np.all(np.diff(slot[kept]) > 0)              # rises with t
                if dropped.size:
                    assert kept.max() < dropped.min()
            elif dropped.size and kept.size:
                assert g[kept].min() >= g[dropped].max()


def test_zero_router_keeps_first_C_tokens():
    # W_g = 0, cf = 1: every token goes to expert 0 and exactly 0..C-1 are kept
    T, N, d = 40, 4, 8
    x = np.random.default_rng(10).standard_normal((T, d))
    r = O.route(x, np.zeros((N, d)))
    C = O.capacity(T, N, 1.0)
    for mode in (O.TOKEN_ORDER, O.GATE_PRIORITY):
        slot, drop, counts = O.assign_slots(r["expert_id"], r["gate"], N, C, mode)
        assert np.array_equal(slot[:C], np.arange(C))
        assert np.all(slot[C:] == -1)
        assert list(counts) == [T, 0, 0, 0]


def test_no_drops_when_cf_at_least_N():
    rng = np.random.default_rng(11)
    for _ in range(20):
        N = int(rng.integers(1, 9))
        T = int(rng.integers(1, 300))
        C = O.capacity(T, N, float(N) + rng.random())
        e = rng.integers(0, N, size=T)
        for mode in (O.TOKEN_ORDER, O.GATE_PRIORITY):
            _, drop, _ = O.assign_slots(e, rng.random(T), N, C, mode)
            assert drop.sum() == 0


def test_batch_composition_dependence():
    # With C fixed, appending tokens never changes earlier tokens in token
    # order; in gate priority a later, higher-gate token can evict one.
    rng = np.random.default_rng(12)
    for _ in range(30):
        N, T0, T1, C = 3, 30, 50, 6
        e = rng.integers(0, N, size=T0 + T1)
        g = rng.random(T0 + T1)
        s0, _, _ = O.assign_slots(e[:T0], g[:T0], N, C, O.TOKEN_ORDER)
        s1, _, _ = O.assign_slots(e, g, N, C, O.TOKEN_ORDER)
        assert np.array_equal(s0, s1[:T0])
    e = np.array([0, 0, 0])
    g = np.array([0.5, 0.4, 0.9])
    s0, _, _ = O.assign_slots(e[:2], g[:2], 1, 2, O.GATE_PRIORITY)
    s1, _, _ = O.assign_slots(e, g, 1, 2, O.GATE_PRIORITY)
    assert list(s0) == [0, 1] and list(s1) == [1, -1, 0]
    # through the real capacity, C grows with T: token order only gains keeps
    for _ in range(30):
        e = rng.integers(0, 4, size=80)
        g = rng.random(80)
        a, _, _ = O.assign_slots(e[:40], g[:40], 4, O.capacity(40, 4, 1.0))
        b, _, _ = O.assign_slots(e, g, 4, O.capacity(80, 4, 1.0))
        assert np.all((a[:40] < 0) | (b[:40] >= 0))


# ---------------------------------------------------------------- expert FFN
def test_expert_ffn_permutation_closed_form():
    # W1 = permutation P, W2 = signed permutation Q: o = Q relu(P x), by indexing
    rng = np.random.default_rng(13)
    n = 7
    pi = rng.permutation(n)
    sigma = rng.permutation(n)
    sgn = rng.choice([-1.0, 2.0], size=n)
    W1 = np.zeros((n, n))
    W1[np.arange(n), pi] = 1.0            # (W1 x)_f = x[pi[f]]
    W2 = np.zeros((n, n))
    W2[np.arange(n), sigma] = sgn         # (W2 h)_j = sgn_j * h[sigma[j]]
    x = rng.standard_normal((9, n))
    o = O.expert_ffn(x, W1, W2)
    h = np.maximum(x[:, pi], 0.0)
    np.testing.assert_array_equal(o, sgn[None, :] * h[:, sigma])


def test_expert_ffn_rectangular_against_torch():
    rng = np.random.default_rng(14)
    d, F = 12, 40
    x = rng.standard_normal((17, d))
    W1 = rng.standard_normal((F, d))
    W2 = rng.standard_normal((d, F))
    tx, t1, t2 = (torch.from_numpy(a) for a in (x, W1, W2))
    ref = torch.nn.functional.linear(torch.relu(torch.nn.functional.linear(tx, t1)), t2).numpy()
    np.testing.assert_allclose(O.expert_ffn(x, W1, W2), ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- whole layer
@pytest.mark.parametrize("gm", [0, 1])
def test_single_expert_is_dense_ffn(gm):
    # N = 1, cf >= 1: C >= T, gate = softmax of one logit = 1 exactly
    rng = np.random.default_rng(15)
    T, d, F = 33, 10, 24
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((1, d))
    W1 = rng.standard_normal((1, F, d))
    W2 = rng.standard_normal((1, d, F))
    out = O.forward(x, Wg, W1, W2, 1.0, gate_multiply=gm)
    assert np.all(out["gate"] == 1.0) and out["drop"].sum() == 0
    tx = torch.from_numpy(x)
    ref = torch.nn.functional.linear(
        torch.relu(torch.nn.functional.linear(tx, torch.from_numpy(W1[0]))),
        torch.from_numpy(W2[0])).numpy()
    np.testing.assert_allclose(out["y"], ref, rtol=1e-12, atol=1e-12)
    assert out["aux_loss"] == pytest.approx(1.0, abs=1e-15)


def test_gate_flag_drop_and_shared():
    rng = np.random.default_rng(16)
    T, d, F, N = 50, 6, 10, 3
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((N, d))
    W1 = rng.standard_normal((N, F, d))
    W2 = rng.standard_normal((N, d, F))
    W1s = rng.standard_normal((F, d))
    W2s = rng.standard_normal((d, F))
    a = O.forward(x, Wg, W1, W2, 0.5, gate_multiply=1)
    b = O.forward(x, Wg, W1, W2, 0.5, gate_multiply=0)
    c = O.forward(x, Wg, W1, W2, 0.5, gate_multiply=1, W1s=W1s, W2s=W2s)
    assert a["drop"].sum() > 0
    for t in range(T):
        if a["drop"][t]:
            assert np.all(a["y"][t] == 0.0) and np.all(b["y"][t] == 0.0)
        else:
            e = a["expert_id"][t]
            o = W2[e] @ np.maximum(W1[e] @ x[t], 0)
            np.testing.assert_allclose(b["y"][t], o, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(a["y"][t], a["gate"][t] * o, rtol=1e-12, atol=1e-12)
        S = W2s @ np.maximum(W1s @ x[t], 0)
        np.testing.assert_allclose(c["y"][t] - a["y"][t], S, rtol=1e-10, atol=1e-10)


def test_expert_relabelling_equivariance():
    rng = np.random.default_rng(17)
    T, d, F, N = 64, 8, 12, 5
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((N, d))
    W1 = rng.standard_normal((N, F, d))
    W2 = rng.standard_normal((N, d, F))
    perm = rng.permutation(N)
    a = O.forward(x, Wg, W1, W2, 1.0)
    b = O.forward(x, Wg[perm], W1[perm], W2[perm], 1.0)
    inv = np.argsort(perm)
    assert np.array_equal(inv[a["expert_id"]], b["expert_id"])
    assert np.array_equal(a["counts"][perm], b["counts"])
    assert np.array_equal(a["slot"], b["slot"])
    np.testing.assert_allclose(a["y"], b["y"], rtol=1e-13, atol=1e-13)
    assert a["aux_loss"] == pytest.approx(b["aux_loss"], rel=1e-13)


def test_forward_rows_matches_forward():
    rng = np.random.default_rng(18)
    T, d, F, N = 90, 8, 16, 4
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((N, d))
    W1 = rng.standard_normal((N, F, d))
    W2 = rng.standard_normal((N, d, F))
    W1s = rng.standard_normal((F, d))
    W2s = rng.standard_normal((d, F))
    full = O.forward(x, Wg, W1, W2, 0.75, O.GATE_PRIORITY, W1s=W1s, W2s=W2s)
    rows = rng.choice(T, 25, replace=False)
    part = O.forward_rows(rows, x, full["expert_id"], full["gate"], full["slot"], 1,
                          lambda e: (W1[e], W2[e]), W1s, W2s)
    np.testing.assert_allclose(part, full["y"][rows], rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ Expanded Drop
def _golden_expanded():
    rows, cands, N, C = [], None, 0, 0
    for line in open(os.path.join(GOLDEN, "expanded_drop.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        if line.startswith("cands"):
            f = line.split()
            N, C = int(f[1].split("=")[1]), int(f[2].split("=")[1])
            cands = np.array([[int(v) for v in c.split(",")] for c in f[3:]])
            continue
        k, e, s, u = (part.split() for part in line.split("|"))
        rows.append((cands, N, C, int(k[0]), [int(v) for v in e], [int(v) for v in s],
                     [int(v) for v in u]))
    return rows


@pytest.mark.parametrize("case", _golden_expanded(),
                         ids=lambda c: f"N{c[1]}C{c[2]}k{c[3]}")
def test_expanded_drop_golden(case):
    cands, N, C, k, want_e, want_s, want_u = case
    e, s, drop, used = O.assign_slots_expanded(cands[:, :k], N, C)
    assert e.tolist() == want_e and s.tolist() == want_s and used.tolist() == want_u
    assert drop.tolist() == [int(v < 0) for v in want_s]


def test_candidates_order_and_ties():
    rng = np.random.default_rng(3)
    l = rng.integers(-2, 3, size=(200, 6)).astype(np.float64)   # many exact ties
    c = O.candidates(l, 6)
    for t in range(l.shape[0]):
        want = sorted(range(6), key=lambda i: (-l[t, i], i))    # logit desc, index asc
        assert c[t].tolist() == want
    # the first candidate is the top-1 expert of the forward
    e, _ = O.top1(l, O.softmax(l))
    assert np.array_equal(c[:, 0], e)


def test_expanded_drop_k1_is_top1_token_order():
    rng = np.random.default_rng(4)
    for T, N, C in [(300, 5, 40), (64, 8, 3), (50, 2, 30)]:
        l = rng.normal(size=(T, N))
        c = O.candidates(l, 1)
        e, s, d, used = O.assign_slots_expanded(c, N, C)
        s0, d0, counts = O.assign_slots(c[:, 0], np.ones(T), N, C, O.TOKEN_ORDER)
        assert np.array_equal(s, s0) and np.array_equal(d, d0)
        assert np.array_equal(used, np.minimum(counts, C)) and np.array_equal(e, c[:, 0])


def test_expanded_drop_invariants():
    rng = np.random.default_rng(5)
    for T, N, C in [(400, 6, 50), (128, 4, 20), (1000, 16, 40), (37, 3, 1)]:
        l = rng.normal(size=(T, N)) + np.linspace(0, 2, N)   # skewed towards high experts
        prev_drops = None
        for k in range(1, N + 1):
            c = O.candidates(l, k)
            e, s, d, used = O.assign_slots_expanded(c, N, C)
            assert np.all(used <= C)
            for i in range(N):   # each expert's slots are 0 .. used - 1, once each
                assert sorted(s[(e == i) & (s >= 0)].tolist()) == list(range(used[i]))
            kept = s >= 0
            # a kept token runs on one of its first k candidates; a dropped
            # token found every one of them full
            assert all(e[t] in c[t].tolist() for t in np.nonzero(kept)[0])
            assert all(used[c[t]].min() == C for t in np.nonzero(~kept)[0])
            drops = int(d.sum())
            assert prev_drops is None or drops <= prev_drops   # more candidates, fewer drops
            prev_drops = drops
        if N * C >= T:   # with every candidate allowed, nothing is dropped
            assert prev_drops == 0


def test_expanded_drop_no_drops_when_capacity_suffices():
    rng = np.random.default_rng(6)
    T, N = 200, 4
    C = O.capacity(T, N, float(N))   # cf >= N: C >= T
    l = rng.normal(size=(T, N))
    c = O.candidates(l, 3)
    e, s, d, _ = O.assign_slots_expanded(c, N, C)
    assert d.sum() == 0 and np.array_equal(e, c[:, 0])   # all placed in pass 1


def test_forward_expanded_reroutes_with_candidate_gate():
    rng = np.random.default_rng(7)
    T, d, F, N = 96, 16, 24, 4
    x = torch.tensor(rng.normal(size=(T, d)))
    W_g = torch.tensor(rng.normal(size=(N, d)) * 0.5)
    W_g[0] += 0.8   # expert 0 over-full
    W1 = torch.tensor(rng.normal(size=(N, F, d)) / np.sqrt(d))
    W2 = torch.tensor(rng.normal(size=(N, d, F)) / np.sqrt(F))
    base = O.forward(x, W_g, W1, W2, 1.0)
    ex = O.forward(x, W_g, W1, W2, 1.0, expand=2)
    assert ex["drop"].sum() < base["drop"].sum()
    assert ex["aux_loss"] == base["aux_loss"] and np.array_equal(ex["counts"], base["counts"])
    moved = np.nonzero((base["drop"] == 1) & (ex["drop"] == 0))[0]
    assert moved.size > 0
    c2 = O.candidates(base["logits"], 2)
    for t in moved:
        e = int(c2[t, 1])
        assert ex["expert_id"][t] == e
        assert ex["gate"][t] == base["probs"][t, e]
        h = torch.relu(x[t] @ W1[e].T)                         # library routines, float64
        assert np.allclose(ex["y"][t], (base["probs"][t, e] * (h @ W2[e].T)).numpy(),
                           rtol=1e-12, atol=1e-12)
    same = np.nonzero(base["drop"] == 0)[0]                  # pass-1 tokens are untouched
    assert np.array_equal(ex["y"][same], base["y"][same])


# ------------------------------------------------------------------ Top-2
def _golden_top2():
    slots, gates, cands, N = [], [], None, 0
    for line in open(os.path.join(GOLDEN, "top2.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        if line.startswith("chosen"):
            f = line.split()
            N = int(f[1].split("=")[1])
            cands = np.array([[int(v) for v in c.split(",")] for c in f[2:]])
        elif line.startswith("gates"):
            lg, ch, g, gr = (part.split() for part in line[len("gates"):].split("|"))
            logits = [math.log(float(v[2:])) if v.startswith("ln") else float(v)
                      for v in lg[0].split(",")]
            gates.append((np.array([logits]), [int(v) for v in ch], [float(v) for v in g],
                          [float(v) for v in gr]))
        else:
            c, s0, s1, u = (part.split() for part in line.split("|"))
            slots.append((cands, N, int(c[0]), [int(v) for v in s0], [int(v) for v in s1],
                          [int(v) for v in u]))
    return slots, gates


@pytest.mark.parametrize("case", _golden_top2()[0], ids=lambda c: f"C{c[2]}")
def test_top2_slots_golden(case):
    cands, N, C, want0, want1, want_u = case
    slot, drop, used = O.assign_slots_top2(cands, N, C)
    assert slot[:, 0].tolist() == want0 and slot[:, 1].tolist() == want1
    assert used.tolist() == want_u
    assert np.array_equal(drop, (slot < 0).astype(np.uint8))


@pytest.mark.parametrize("case", _golden_top2()[1], ids=lambda c: str(c[1]))
def test_top2_gates_golden(case):
    logits, chosen, g, gr = case
    c = O.candidates(logits, 2)
    assert c[0].tolist() == chosen
    p = O.softmax(logits)
    np.testing.assert_allclose(O.top2_gates(p, c, 0)[0], g, rtol=1e-15)
    np.testing.assert_allclose(O.top2_gates(p, c, 1)[0], gr, rtol=1e-15)


def test_top2_first_choices_are_the_top1_assignment():
    rng = np.random.default_rng(11)
    for T, N, C in [(300, 5, 40), (64, 8, 3), (500, 16, 20)]:
        l = rng.normal(size=(T, N)) + np.linspace(0, 1.5, N)
        c = O.candidates(l, 2)
        slot, _, _ = O.assign_slots_top2(c, N, C)
        s0, _, counts = O.assign_slots(c[:, 0], np.ones(T), N, C, O.TOKEN_ORDER)
        assert np.array_equal(slot[:, 0], s0)
        # every second choice an expert keeps sits after all of its kept first choices
        for i in range(N):
            second = slot[(c[:, 1] == i) & (slot[:, 1] >= 0), 1]
            assert np.all(second >= min(counts[i], C))


def test_top2_invariants():
    rng = np.random.default_rng(12)
    for T, N, C in [(400, 6, 50), (128, 4, 20), (1000, 16, 40), (37, 3, 1), (50, 2, 60)]:
        l = rng.normal(size=(T, N)) + np.linspace(0, 2, N)
        c = O.candidates(l, 2)
        assert np.all(c[:, 0] != c[:, 1])
        slot, drop, used = O.assign_slots_top2(c, N, C)
        assert np.all(used <= C)
        for i in range(N):   # both choices together fill slots 0 .. used - 1 once each
            s = np.concatenate([slot[(c[:, r] == i) & (slot[:, r] >= 0), r] for r in range(2)])
            assert sorted(s.tolist()) == list(range(used[i]))
            for r in range(2):   # token order within a pass
                sr = slot[(c[:, r] == i) & (slot[:, r] >= 0), r]
                assert np.all(np.diff(sr) > 0)
        if 2 * T <= C:
            assert drop.sum() == 0
        p = O.softmax(l)
        g = O.top2_gates(p, c, 0)
        assert np.all(g[:, 0] >= g[:, 1]) and np.all(g.sum(axis=1) <= 1 + 1e-15)
        np.testing.assert_allclose(O.top2_gates(p, c, 1).sum(axis=1), 1.0, rtol=1e-15)


def test_top2_brute_force_definition():
    """Kept iff fewer than C earlier (pass-major, then token order) choices
    hold the same expert: the O(T^2) definition, over every assignment of
    ordered expert pairs for small T."""
    N = 3
    pairs = [(a, b) for a in range(N) for b in range(N) if a != b]
    rng = np.random.default_rng(13)
    for T in (1, 2, 3, 4):
        combos = list(itertools.product(pairs, repeat=T))
        if len(combos) > 400:
            combos = [combos[i] for i in rng.choice(len(combos), 400, replace=False)]
        for combo in combos:
            c = np.array(combo)
            order = [(r, t) for r in range(2) for t in range(T)]
            for C in range(1, 2 * T + 1):
                slot, _, _ = O.assign_slots_top2(c, N, C)
                for k, (r, t) in enumerate(order):
                    before = sum(1 for (r2, t2) in order[:k] if c[t2, r2] == c[t, r])
                    # slot = number of earlier choices the expert kept
                    want = before if before < C else -1
                    assert slot[t, r] == want


def test_forward_top2_identical_experts_closed_form():
    """All experts equal, nothing dropped: y = (g0 + g1) E(x); with
    renormalised gates that is E(x) itself (checked against torch float64)."""
    rng = np.random.default_rng(14)
    T, d, F, N = 40, 12, 20, 5
    x = torch.tensor(rng.normal(size=(T, d)))
    W_g = torch.tensor(rng.normal(size=(N, d)))
    w1 = torch.tensor(rng.normal(size=(F, d)) / np.sqrt(d))
    w2 = torch.tensor(rng.normal(size=(d, F)) / np.sqrt(F))
    W1, W2 = w1.expand(N, F, d).clone(), w2.expand(N, d, F).clone()
    E = torch.nn.functional.linear(torch.relu(torch.nn.functional.linear(x, w1)), w2).numpy()
    cf = float(2 * N)   # C >= 2T: both choices of every token fit
    out = O.forward_top2(x, W_g, W1, W2, cf, gate_multiply=1, renormalize=1)
    assert out["drop"].sum() == 0
    np.testing.assert_allclose(out["y"], E, rtol=1e-12, atol=1e-12)
    out = O.forward_top2(x, W_g, W1, W2, cf, gate_multiply=1, renormalize=0)
    p = torch.softmax(x @ W_g.T, dim=1).numpy()
    top2 = np.sort(p, axis=1)[:, -2:].sum(axis=1)
    np.testing.assert_allclose(out["y"], top2[:, None] * E, rtol=1e-12, atol=1e-12)
    out = O.forward_top2(x, W_g, W1, W2, cf, gate_multiply=0)
    np.testing.assert_allclose(out["y"], 2 * E, rtol=1e-12, atol=1e-12)


def test_forward_top2_zero_second_expert_is_top1():
    """N = 2 with expert 0 always first: choice 1 is expert 1; with W of
    expert 1 zero the layer is the top-1 layer with the same gate."""
    rng = np.random.default_rng(15)
    T, d, F = 30, 8, 16
    x = torch.tensor(rng.normal(size=(T, d)))
    W_g = torch.tensor(rng.normal(size=(2, d)) * 0.1)
    b_g = torch.tensor([5.0, 0.0])
    W1 = torch.tensor(rng.normal(size=(2, F, d)))
    W2 = torch.tensor(rng.normal(size=(2, d, F)))
    W1[1] = 0
    for cf in (0.5, 2.0):
        a = O.forward_top2(x, W_g, W1, W2, cf, gate_multiply=1, b_g=b_g)
        b = O.forward(x, W_g, W1, W2, cf, gate_multiply=1, b_g=b_g)
        assert np.all(a["expert_id"][:, 0] == 0)
        np.testing.assert_allclose(a["y"], b["y"], rtol=1e-13, atol=1e-13)
        assert np.array_equal(a["slot"][:, 0], b["slot"])
        assert a["aux_loss"] == b["aux_loss"]


def test_forward_rows_top2_matches_forward_top2():
    rng = np.random.default_rng(16)
    T, d, F, N = 80, 8, 12, 6
    x = torch.tensor(rng.normal(size=(T, d)))
    W_g = torch.tensor(rng.normal(size=(N, d)))
    W1 = torch.tensor(rng.normal(size=(N, F, d)))
    W2 = torch.tensor(rng.normal(size=(N, d, F)))
    W1s = torch.tensor(rng.normal(size=(F, d)))
    W2s = torch.tensor(rng.normal(size=(d, F)))
    full = O.forward_top2(x, W_g, W1, W2, 0.7, gate_multiply=1, renormalize=1, W1s=W1s, W2s=W2s)
    assert 0 < full["drop"].sum() < 2 * T
    rows = rng.choice(T, 30, replace=False)
    part = O.forward_rows_top2(rows, x, full["expert_id"], full["gate"], full["slot"], 1,
                               lambda e: (W1[e], W2[e]), W1s, W2s)
    np.testing.assert_allclose(part, full["y"][rows], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ Expert choice
def _golden_expert_choice():
    rows, scores = [], None
    for line in open(os.path.join(GOLDEN, "expert_choice.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        if line.startswith("scores"):
            f = line.split()
            scores = np.array([[float(v) for v in c.split(",")] for c in f[2:]])
            continue
        c, e0, e1, per = (part.split() for part in line.split("|"))
        rows.append((scores, int(c[0]), [int(v) for v in e0], [int(v) for v in e1],
                     [int(v) for v in per]))
    return rows


@pytest.mark.parametrize("case", _golden_expert_choice(), ids=lambda c: f"C{c[1]}")
def test_expert_choice_golden(case):
    scores, C, want0, want1, want_per = case
    chosen, gates = O.expert_choice(scores, C)
    assert chosen[0].tolist() == want0 and chosen[1].tolist() == want1
    assert np.bincount(chosen.ravel(), minlength=scores.shape[0]).tolist() == want_per
    for e in range(2):
        assert np.array_equal(gates[e], scores[chosen[e], e])


def test_expert_choice_brute_force_definition():
    """Token t is in expert e's list iff fewer than C tokens beat it
    (higher score, or equal score and lower index); its slot is that number."""
    rng = np.random.default_rng(21)
    for T, N in [(7, 3), (12, 2), (30, 5)]:
        s = rng.integers(0, 4, size=(T, N)).astype(np.float64)   # many ties
        for C in range(1, T + 2):
            chosen, _ = O.expert_choice(s, C)
            for e in range(N):
                for t in range(T):
                    beat = sum(1 for u in range(T)
                               if s[u, e] > s[t, e] or (s[u, e] == s[t, e] and u < t))
                    if beat < C:
                        assert chosen[e, beat] == t
                    else:
                        assert t not in chosen[e].tolist()


def test_expert_choice_invariants():
    rng = np.random.default_rng(22)
    T, N = 300, 8
    p = O.softmax(rng.normal(size=(T, N)))
    for C in (1, 10, 37, 300, 400):
        chosen, gates = O.expert_choice(p, C)
        assert chosen.shape == (N, min(C, T))
        for e in range(N):
            assert len(set(chosen[e].tolist())) == min(C, T)          # no token twice
            assert np.all(np.diff(gates[e]) <= 0)                     # best first
            rest = np.setdiff1d(np.arange(T), chosen[e])
            if rest.size:
                assert p[rest, e].max() <= gates[e].min()              # nobody left is better
        per = np.bincount(chosen.ravel(), minlength=T)
        assert per.sum() == N * min(C, T) and per.max() <= N


def test_forward_expert_choice_closed_forms():
    """C >= T: every expert takes every token, y = sum_e s[t, e] E_e(x); with
    identical experts that is E(x) (scores sum to 1) and N E(x) unscaled."""
    rng = np.random.default_rng(23)
    T, d, F, N = 24, 10, 16, 4
    x = torch.tensor(rng.normal(size=(T, d)))
    W_g = torch.tensor(rng.normal(size=(N, d)))
    w1 = torch.tensor(rng.normal(size=(F, d)) / np.sqrt(d))
    w2 = torch.tensor(rng.normal(size=(d, F)) / np.sqrt(F))
    W1, W2 = w1.expand(N, F, d).clone(), w2.expand(N, d, F).clone()
    E = torch.nn.functional.linear(torch.relu(torch.nn.functional.linear(x, w1)), w2).numpy()
    out = O.forward_expert_choice(x, W_g, W1, W2, float(N), gate_multiply=1)
    assert np.all(out["experts_per_token"] == N)
    np.testing.assert_allclose(out["y"], E, rtol=1e-12, atol=1e-12)
    out = O.forward_expert_choice(x, W_g, W1, W2, float(N), gate_multiply=0)
    np.testing.assert_allclose(out["y"], N * E, rtol=1e-12, atol=1e-12)
    # cf small: tokens nobody took get exactly zero
    out = O.forward_expert_choice(x, W_g, W1, W2, 0.25, gate_multiply=1)
    none = out["experts_per_token"] == 0
    assert none.any() and np.all(out["y"][none] == 0)


def test_forward_rows_expert_choice_matches_forward():
    rng = np.random.default_rng(24)
    T, d, F, N = 60, 8, 12, 5
    x = torch.tensor(rng.normal(size=(T, d)))
    W_g = torch.tensor(rng.normal(size=(N, d)))
    W1 = torch.tensor(rng.normal(size=(N, F, d)))
    W2 = torch.tensor(rng.normal(size=(N, d, F)))
    W1s = torch.tensor(rng.normal(size=(F, d)))
    W2s = torch.tensor(rng.normal(size=(d, F)))
    full = O.forward_expert_choice(x, W_g, W1, W2, 1.3, W1s=W1s, W2s=W2s)
    rows = rng.choice(T, 25, replace=False)
    part = O.forward_rows_expert_choice(rows, x, full["chosen"], full["gates"], 1,
                                        lambda e: (W1[e], W2[e]), W1s, W2s)
    np.testing.assert_allclose(part, full["y"][rows], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ backward
def _loss(x, W_g, W1, W2, cf, dy, mode, gm, b_g, W1s, W2s, alpha):
    f = O.forward(x, W_g, W1, W2, cf, mode, gm, b_g, W1s, W2s)
    return float(np.sum(f["y"] * dy.numpy()) + alpha * f["aux_loss"]), f


@pytest.mark.parametrize("mode,gm,shared,cf", [(0, 1, 0, 0.8), (1, 1, 1, 0.8), (0, 0, 0, 1.5),
                                               (1, 0, 1, 0.6)])
def test_backward_matches_central_differences(mode, gm, shared, cf):
    """Every gradient of <dy, y> + alpha * L_aux against central differences
    of the (pinned) forward, at entries whose perturbation leaves the
    routing unchanged."""
    rng = np.random.default_rng(31 + 2 * mode + gm)
    T, d, F, N, alpha = 24, 6, 10, 3, 0.37
    x = torch.tensor(rng.normal(size=(T, d)))
    W_g = torch.tensor(rng.normal(size=(N, d)))
    b_g = torch.tensor(rng.normal(size=N) * 0.3)
    W1 = torch.tensor(rng.normal(size=(N, F, d)))
    W2 = torch.tensor(rng.normal(size=(N, d, F)))
    W1s = torch.tensor(rng.normal(size=(F, d))) if shared else None
    W2s = torch.tensor(rng.normal(size=(d, F))) if shared else None
    dy = torch.tensor(rng.normal(size=(T, d)))
    g = O.backward(x, W_g, W1, W2, cf, dy, mode, gm, b_g, W1s, W2s, aux_coef=alpha)
    fw = g["forward"]
    assert 0 < fw["drop"].sum() < T or cf > 1
    params = {"x": x, "W_g": W_g, "b_g": b_g, "W1": W1, "W2": W2}
    grads = {"x": g["dx"], "W_g": g["dW_g"], "b_g": g["db_g"], "W1": g["dW1"], "W2": g["dW2"]}
    if shared:
        params.update(W1s=W1s, W2s=W2s)
        grads.update(W1s=g["dW1s"], W2s=g["dW2s"])
    eps, checked = 1e-6, 0
    for name, tns in params.items():
        flat = tns.view(-1)
        for idx in rng.choice(flat.numel(), min(12, flat.numel()), replace=False):
            old = float(flat[idx])
            vals = []
            for s in (1.0, -1.0):
                flat[idx] = old + s * eps
                a = dict(params)
                lv, f2 = _loss(a["x"], a["W_g"], a["W1"], a["W2"], cf, dy, mode, gm, a["b_g"],
                               a.get("W1s"), a.get("W2s"), alpha)
                same = (np.array_equal(f2["expert_id"], fw["expert_id"])
                        and np.array_equal(f2["slot"], fw["slot"]))
                vals.append((lv, same))
            flat[idx] = old
            if not (vals[0][1] and vals[1][1]):
                continue   # the routing moved: no derivative there
            fd = (vals[0][0] - vals[1][0]) / (2 * eps)
            an = float(np.asarray(grads[name]).reshape(-1)[idx])
            assert abs(fd - an) <= 1e-5 * max(1.0, abs(an)), (name, int(idx), fd, an)
            checked += 1
    assert checked >= 40


def test_backward_one_expert_is_the_dense_ffn_gradient():
    """N = 1, nothing dropped: the gate is exactly 1 and the router gets no
    gradient; the FFN gradients are those of a dense two-layer ReLU MLP,
    from torch.autograd in float64."""
    rng = np.random.default_rng(33)
    T, d, F = 16, 5, 9
    x = torch.tensor(rng.normal(size=(T, d)), requires_grad=True)
    W1 = torch.tensor(rng.normal(size=(1, F, d)), requires_grad=True)
    W2 = torch.tensor(rng.normal(size=(1, d, F)), requires_grad=True)
    W_g = torch.tensor(rng.normal(size=(1, d)))
    dy = torch.tensor(rng.normal(size=(T, d)))
    y = torch.nn.functional.linear(torch.relu(torch.nn.functional.linear(x, W1[0])), W2[0])
    (y * dy).sum().backward()
    g = O.backward(x.detach(), W_g, W1.detach(), W2.detach(), 1.0, dy, aux_coef=0.5)
    np.testing.assert_allclose(g["dx"], x.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dW1"], W1.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dW2"], W2.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(g["dW_g"] == 0) and np.all(g["db_g"] == 0)
