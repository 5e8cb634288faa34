"""Pins of the oracle's relaxed thresholds and per-request temperatures (verify variants).

The relaxed rule is pinned by the worked example the pages print for it (acceptance 1.0, total
variation 0.35 on the six-token toy) and by closed forms for one candidate; thresholds of 1 must
reduce to the exact rule; a tree level with several candidates (one at or above
threshold_single, one of probability 0) matches its closed form.  The per-request temperature
dispatch is pinned by the argmax-prefix rule computed here from numpy argmax, and by the
single-temperature oracle on each request.

Planting each of these mistakes in a copy of the oracle fails at least one pin: p(x) times
threshold_acc for p(x) / threshold_acc, threshold_single ignored (chain and tree), a candidate's
own p for the running sum, threshold_acc ignored in trees, a running sum carried into a level,
the first request's temperature used for every request, the draft emitted at a greedy stop, a
greedy request accepting past its first mismatch.
Dropping the p > 0 guard of an acceptance is not caught and cannot be: with thresholds in (0, 1]
a candidate of probability 0 meets neither condition on a coin that an earlier one left."""
import json
import os

import numpy as np
import pytest

G = 1024


def test_relaxed_thresholds_toy(oracle, golden_dir):
    toy = json.load(open(os.path.join(golden_dir, "toy_six_token_relaxed.json")))
    P, Q = np.array(toy["P"]), np.array(toy["Q"])
    cand = list(np.argsort(-Q, kind="stable")[:3])
    assert cand == [1, 3, 0]
    dist, acc = oracle.grid_tree_first_token(P, cand, G, toy["threshold_single"], toy["threshold_acc"])
    assert acc == pytest.approx(toy["acceptance"], abs=1e-12)
    tv = 0.5 * np.abs(dist - P).sum()
    assert tv == pytest.approx(toy["total_variation"], abs=2.0 / G)
    # The emitted mass sits on the candidates only (every coin accepts one of them).
    assert dist[[2, 4, 5]].sum() == pytest.approx(0.0, abs=1e-12)


def test_thresholds_of_one_are_the_exact_rule(oracle):
    rng = np.random.default_rng(0)
    for _ in range(200):
        V, k = int(rng.integers(2, 9)), int(rng.integers(1, 5))
        p = rng.dirichlet(np.ones(V) * 0.5, size=k + 1)
        d = rng.integers(0, V, k).astype(np.int32)
        if rng.random() < 0.2:
            d[rng.integers(0, k)] = -1
        u, v = rng.random(k + 1), rng.random(k + 1)
        a = oracle.chain_core(p, None, d, u, v)
        b = oracle.chain_core(p, None, d, u, v, 0.999999, 1.0)
        c = oracle.chain_core(p, None, d, u, v, 1.0, 1.0)
        assert a["tokens"].tolist() == c["tokens"].tolist() and a["accept_len"] == c["accept_len"]
        # A threshold just below 1 changes nothing unless some p(x) reaches it.
        if all(p[i, d[i]] < 0.999999 for i in range(k) if d[i] >= 0):
            assert b["tokens"].tolist() == c["tokens"].tolist()
    P = rng.dirichlet(np.ones(7))
    dist, acc = oracle.grid_tree_first_token(P, [3, 1], G, 1.0, 1.0)
    np.testing.assert_allclose(dist, P, atol=2.0 / G)
    assert acc == pytest.approx(P[3] + P[1], abs=2.0 / G)


@pytest.mark.parametrize("thr_single,thr_acc", [(1.0, 0.5), (0.3, 1.0), (0.2, 0.7)])
def test_relaxed_single_candidate_closed_form(oracle, thr_single, thr_acc):
    """One candidate x: accepted with probability min(1, p(x) / thr_acc), or always when
    p(x) >= thr_single; otherwise the draw comes from p with x zeroed (the exact residual)."""
    rng = np.random.default_rng(1)
    for _ in range(6):
        V = 5
        p = rng.dirichlet(np.ones(V))
        x = int(rng.integers(0, V))
        px = p[x]
        want = 1.0 if px >= thr_single else min(1.0, px / thr_acc)
        us = (np.arange(256) + 0.5) / 256
        got = np.mean([oracle.chain_core(np.stack([p, p]), None, np.array([x], np.int32),
                                         np.array([u, 0.5]), np.array([0.5, 0.5]),
                                         thr_single, thr_acc)["accept_len"] == 1 for u in us])
        assert got == pytest.approx(want, abs=1.0 / 256 + 1e-12)
        # A rejected candidate is never emitted at that slot.
        r = oracle.chain_core(np.stack([p, p]), None, np.array([x], np.int32),
                              np.array([0.9999, 0.5]), np.array([0.3, 0.5]), thr_single, thr_acc)
        if r["accept_len"] == 0:
            assert r["tokens"][0] != x


def _relaxed_level(p, children, ts, ta):
    """One tree level under the relaxed rule, in closed form: children are tried in order, child
    j (p_j > 0) accepting a coin below S_j / ta (S_j the running sum of the tried children's p)
    or any coin when p_j >= ts; the first acceptance wins.  Returns the first token's law."""
    dist = np.zeros_like(p)
    prev, S = 0.0, 0.0
    for t in children:
        S += p[t]
        if p[t] <= 0.0:
            continue
        hi = 1.0 if p[t] >= ts else min(1.0, S / ta)
        dist[t] += max(0.0, hi - prev)
        prev = max(prev, hi)
    rest = np.ones_like(p, dtype=bool)
    rest[list(children)] = False
    if rest.any() and p[rest].sum() > 0:
        dist[rest] = (1.0 - prev) * p[rest] / p[rest].sum()
    return dist, prev


@pytest.mark.parametrize("ts,ta", [(0.25, 1.0), (0.4, 0.8), (1.0, 0.6), (0.2, 0.3)])
def test_relaxed_tree_level_closed_form(oracle, ts, ta):
    """Several candidates, one of them at or above threshold_single, one of probability 0: the
    grid-integrated first token matches the closed form above."""
    rng = np.random.default_rng(3)
    for _ in range(5):
        V = 7
        p = rng.dirichlet(np.ones(V))
        p[4] = 0.0
        if ts < 1.0:  # child 2 at threshold_single + 0.05, the rest scaled around it
            others = np.arange(V) != 2
            p[others] *= (1.0 - (ts + 0.05)) / p[others].sum()
            p[2] = ts + 0.05
        p /= p.sum()
        assert ts >= 1.0 or p[2] >= ts
        children = [0, 4, 2, 5]
        dist, acc = oracle.grid_tree_first_token(p, children, G, ts, ta)
        want, wacc = _relaxed_level(p, children, ts, ta)
        assert acc == pytest.approx(wacc, abs=2.0 / G)
        np.testing.assert_allclose(dist, want, atol=3.0 / G)


def _argmax_prefix(lg, d):
    am = lg.argmax(-1)
    j = 0
    while j < len(d) and d[j] >= 0 and d[j] == am[j]:
        j += 1
    return j, [int(t) for t in d[:j]] + [int(am[j])]


def test_mixed_temperatures_chain(oracle):
    rng = np.random.default_rng(2)
    B, k, V = 10, 4, 61
    lg = rng.normal(0, 2.0, (B, k + 1, V))
    am = lg.argmax(-1)
    d = np.where(rng.random((B, k)) < 0.6, am[:, :k], rng.integers(0, V, (B, k))).astype(np.int32)
    temps = np.array([0.0, 1.0, 0.7, 0.0, 2.0, 1.3, 0.0, 0.5, 1.0, 0.0])
    r = oracle.verify_ex(lg, d, None, temps, seed=9, offset=4)
    for b in range(B):
        if temps[b] == 0.0:
            j, toks = _argmax_prefix(lg[b], d[b])
            assert r["accept_len"][b] == j
            assert r["out_tokens"][b, : j + 1].tolist() == toks
            assert (r["out_tokens"][b, j + 1:] == -1).all()
            assert not r["out_probs"][b].any()
        else:
            ref = oracle.verify_rejection(lg, d, None, temps[b], 9, 4, req_ids=[b])
            assert r["accept_len"][b] == ref["accept_len"][0]
            assert r["out_tokens"][b].tolist() == ref["out_tokens"][0].tolist()
            np.testing.assert_array_equal(r["out_probs"][b], ref["out_probs"][0])
    # One temperature for all equals the single-temperature entry point.
    r1 = oracle.verify_ex(lg, d, None, np.full(B, 0.8), 9, 4)
    r2 = oracle.verify_rejection(lg, d, None, 0.8, 9, 4)
    np.testing.assert_array_equal(r1["out_tokens"], r2["out_tokens"])
    # With draft probabilities the sampled requests follow the standard rule at their T.
    q = rng.dirichlet(np.ones(V), size=(B, k)).astype(np.float32)
    r = oracle.verify_ex(lg, d, q, temps, 9, 4)
    for b in np.flatnonzero(temps > 0):
        ref = oracle.verify_rejection(lg, d, q, temps[b], 9, 4, req_ids=[b])
        assert r["out_tokens"][b].tolist() == ref["out_tokens"][0].tolist()


def test_mixed_temperatures_tree(oracle):
    rng = np.random.default_rng(3)
    B, N, V = 8, 7, 41
    lg = rng.normal(0, 2.0, (B, N, V))
    parents = np.zeros((B, N), np.int32)
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        parents[b, 0], tokens[b, 0] = -1, -1
        for j in range(1, N):
            parents[b, j] = rng.integers(0, j)
            tokens[b, j] = lg[b, parents[b, j]].argmax() if rng.random() < 0.6 else rng.integers(0, V)
        # siblings must differ for the target-only rule
        for j in range(1, N):
            while any(parents[b, m] == parents[b, j] and tokens[b, m] == tokens[b, j] for m in range(1, j)):
                tokens[b, j] = rng.integers(0, V)
    temps = np.array([0.0, 1.0, 0.0, 0.6, 1.5, 0.0, 1.0, 0.9])
    r = oracle.verify_tree_ex(lg, tokens, parents, temps, seed=5, offset=0)
    for b in range(B):
        if temps[b] == 0.0:
            # Greedy walk from the definition: follow the child whose token is the row's argmax.
            cur, path = 0, []
            while True:
                am = int(lg[b, cur].argmax())
                nxt = [j for j in range(1, N) if parents[b, j] == cur and tokens[b, j] == am]
                if not nxt:
                    break
                cur = nxt[0]
                path.append(cur)
            assert r["accept_len"][b] == len(path)
            assert r["accept_index"][b, 1: len(path) + 1].tolist() == path
            assert r["out_tokens"][b, len(path)] == int(lg[b, cur].argmax())
        else:
            ref = oracle.verify_tree(lg, tokens, parents, 1, temps[b], 5, 0, req_ids=[b])
            assert r["out_tokens"][b].tolist() == ref["out_tokens"][0].tolist()
            assert r["accept_index"][b].tolist() == ref["accept_index"][0].tolist()


def test_invalid_options_are_rejected(oracle):
    lg = np.zeros((2, 3, 5))
    d = np.zeros((2, 2), np.int32)
    with pytest.raises(RuntimeError):
        oracle.verify_ex(lg, d, None, [1.0, -1.0], 0, 0)
    with pytest.raises(RuntimeError):
        oracle.verify_ex(lg, d, None, [1.0, 1.0], 0, 0, thr_single=0.0)
    with pytest.raises(RuntimeError):
        oracle.verify_ex(lg, d, np.full((2, 2, 5), 0.2, np.float32), [1.0, 1.0], 0, 0, thr_acc=0.5)
