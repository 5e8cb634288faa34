"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here compares the oracle with something other than itself: values printed on the
pages (tests/golden), closed forms, exact integration of the decision functions over a grid of
uniforms, library routines for the special cases that reduce to one, and brute force.
"""
import json
import os

import numpy as np
import pytest
from scipy import special, stats

G_FINE = 2048  # grid side for the page's toy case
G = 1024  # grid side for random cases


def _toy(golden_dir):
    return json.load(open(os.path.join(golden_dir, "toy_six_token.json")))


# --------------------------------------------------------------------------------------------
# Single position, exact over a (u, v) grid: the emitted token is distributed as p for any q,
# and the acceptance rate is sum(min(p, q)) ("投机解码", 采样：标准拒绝采样 derivation).
# Each boundary of the step function costs at most 1/G of mass, so the tolerance is (V+1)/G.
# --------------------------------------------------------------------------------------------
def test_toy_standard_rejection(oracle, golden_dir):
    toy = _toy(golden_dir)
    P, Q = np.array(toy["P"]), np.array(toy["Q"])
    dist, acc = oracle.grid_chain_first_token(P, Q, Q, G_FINE)
    assert abs(acc - toy["acceptance"]["standard"]) < 2.0 / G_FINE
    assert np.max(np.abs(dist - P)) < (len(P) + 1) / G_FINE


def test_toy_one_hot(oracle, golden_dir):
    toy = _toy(golden_dir)
    P, Q = np.array(toy["P"]), np.array(toy["Q"])
    x = int(np.argmax(Q))
    w = np.zeros_like(P)
    w[x] = 1.0
    dist, acc = oracle.grid_chain_first_token(P, None, w, G_FINE)
    assert abs(acc - toy["acceptance"]["one_hot"]) < 2.0 / G_FINE
    assert np.max(np.abs(dist - P)) < (len(P) + 1) / G_FINE


def test_toy_tree_target_only(oracle, golden_dir):
    toy = _toy(golden_dir)
    P, Q = np.array(toy["P"]), np.array(toy["Q"])
    children = list(np.argsort(-Q, kind="stable")[:3])
    assert children == [1, 3, 0]
    dist, acc = oracle.grid_tree_first_token(P, children, G_FINE)
    assert abs(acc - toy["acceptance"]["tree_target_only_three_candidates"]) < 2.0 / G_FINE
    assert np.max(np.abs(dist - P)) < (len(P) + 1) / G_FINE


@pytest.mark.parametrize("V,seed", [(2, 0), (3, 1), (5, 2), (6, 3)])
def test_random_pairs_preserve_p(oracle, V, seed):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.full(V, 0.7))
    q = rng.dirichlet(np.full(V, 0.7))
    tol = (V + 1) / G
    # standard: drafts drawn from q
    dist, acc = oracle.grid_chain_first_token(p, q, q, G)
    assert abs(acc - np.minimum(p, q).sum()) < 2.0 / G
    assert np.max(np.abs(dist - p)) < tol
    # one-hot with an arbitrary draft distribution: acceptance is E_w[p(x)]
    w = rng.dirichlet(np.ones(V))
    dist, acc = oracle.grid_chain_first_token(p, None, w, G)
    assert abs(acc - (w * p).sum()) < 2.0 / G
    assert np.max(np.abs(dist - p)) < tol
    # target-only tree with a random candidate set in random order
    m = int(rng.integers(1, V + 1))
    children = list(rng.permutation(V)[:m])
    dist, acc = oracle.grid_tree_first_token(p, children, G)
    assert abs(acc - p[children].sum()) < 2.0 / G
    assert np.max(np.abs(dist - p)) < tol


def test_q_with_zeros_and_p_with_zeros(oracle):
    # q(x) = 0 must accept whenever p(x) > 0 ("投机解码", 对照：mistral.rs); p(x) = 0 never accepts.
    p = np.array([0.5, 0.0, 0.3, 0.2])
    q = np.array([0.0, 0.6, 0.1, 0.3])
    dist, acc = oracle.grid_chain_first_token(p, q, q, G)
    assert abs(acc - np.minimum(p, q).sum()) < 2.0 / G
    assert np.max(np.abs(dist - p)) < 5.0 / G
    P2 = np.stack([p, p])
    for u in (0.0, 0.5, 1.0 - 2 ** -24):
        r = oracle.chain_core(P2, q[None, :], [0], [u, 0.5], [0.5, 0.5])
        assert r["accept_len"] == 1 and r["tokens"][0] == 0
    for u in (0.0, 0.3):
        r = oracle.chain_core(P2, q[None, :], [1], [u, 0.5], [0.5, 0.5])
        assert r["accept_len"] == 0 and r["tokens"][0] != 1


def test_accept_test_is_strict(oracle):
    p = np.array([[0.5, 0.25, 0.25], [1 / 3, 1 / 3, 1 / 3]])
    r = oracle.chain_core(p, None, [0], [0.5, 0.0], [0.0, 0.0])
    assert r["accept_len"] == 0  # u == p(x) rejects
    r = oracle.chain_core(p, None, [0], [0.5 - 2 ** -24, 0.0], [0.0, 0.0])
    assert r["accept_len"] == 1


def test_inverse_cdf_edges(oracle):
    # Row 1 is a bonus row with binary-exact probabilities; C = [.25, .5, 1].
    p = np.array([[1.0, 0.0, 0.0], [0.25, 0.25, 0.5]])
    draw = lambda v: oracle.chain_core(p, None, [0], [0.0, 0.0], [0.0, v])["tokens"][1]
    assert draw(0.0) == 0
    assert draw(0.25 - 2 ** -24) == 0
    assert draw(0.25) == 1  # smallest y with C(y) strictly above v*Z
    assert draw(0.5) == 2
    assert draw(1.0 - 2 ** -24) == 2


def test_absent_draft_draws_from_p(oracle):
    rng = np.random.default_rng(5)
    V = 5
    p = rng.dirichlet(np.ones(V), size=3)
    counts = np.zeros(V)
    for c in range(G):
        r = oracle.chain_core(p, None, [-1, 2], [0.0, 0.0, 0.0], [(c + 0.5) / G, 0.9, 0.9])
        assert r["accept_len"] == 0
        counts[r["tokens"][0]] += 1
        assert r["tokens"][1] == -1 and r["tokens"][2] == -1
    assert np.max(np.abs(counts / G - p[0])) < (V + 1) / G


# --------------------------------------------------------------------------------------------
# Softmax / argmax special cases that reduce to library routines.
# --------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 0.8, 0.3, 2.5])
def test_softmax_matches_library(oracle, T):
    rng = np.random.default_rng(11)
    l32 = (rng.standard_normal((4, 1000)) * 3).astype(np.float32)
    p = oracle.softmax_rows(l32, T)
    ref = special.softmax(l32.astype(np.float64) / T, axis=-1)
    assert np.max(np.abs(p - ref) / ref) < 1e-12
    # bf16 inputs are widened exactly: the same values as float32 give the same p.
    bits = (l32.view(np.uint32) >> 16).astype(np.uint16)
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(oracle.softmax_rows(bits, T), oracle.softmax_rows(widened, T))


def test_argmax_lowest_index_on_ties(oracle):
    l = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0], [-np.inf, 0.0, -1.0, 0.0]])
    assert list(oracle.argmax_rows(l)) == [1, 0, 1]
    rng = np.random.default_rng(3)
    l = np.round(rng.standard_normal((50, 40)) * 2).astype(np.float32)  # many ties
    assert list(oracle.argmax_rows(l)) == list(np.argmax(l, axis=-1))


def test_invalid_rows(oracle):
    B, k, V = 4, 1, 8
    logits = np.zeros((B, k + 1, V))
    logits[0, 0, 3] = np.nan
    logits[1, 1, 2] = np.inf
    logits[2, 0, :] = -np.inf
    logits[3, 0, :5] = -np.inf  # finite entries remain: valid
    drafts = np.zeros((B, k), np.int32)
    r = oracle.verify_rejection(logits, drafts, None, 1.0, 1, 0)
    assert list(r["status"]) == [2, 2, 2, 0]
    assert (r["out_tokens"][:3] == -1).all() and (r["accept_len"][:3] == -1).all()
    g = oracle.verify_greedy(logits, drafts)
    assert list(g["status"]) == [2, 2, 2, 0]


def test_bad_draft_ids(oracle):
    B, k, V = 3, 2, 6
    logits = np.zeros((B, k + 1, V))
    drafts = np.array([[0, 6], [-2, 0], [-1, 5]], np.int32)
    r = oracle.verify_rejection(logits, drafts, None, 1.0, 1, 0)
    assert list(r["status"]) == [1, 1, 0]
    logits[0, 2, 0] = np.nan
    r = oracle.verify_rejection(logits, drafts, None, 1.0, 1, 0)
    assert r["status"][0] == 2  # the largest fault code of the request


# --------------------------------------------------------------------------------------------
# Greedy: DFlash's prefix rule, matches = cand == argmax; correct_len = cumprod(matches).sum;
# bonus = argmax[correct_len] ("The speculative decoding zoo", DFlash section).
# --------------------------------------------------------------------------------------------
def test_greedy_is_argmax_prefix(oracle):
    rng = np.random.default_rng(0)
    B, k, V = 300, 5, 37
    logits = np.round(rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    am = np.argmax(logits, axis=-1)
    drafts = am[:, :k].copy()
    cut = rng.integers(0, k + 1, size=B)
    for b in range(B):
        if cut[b] < k:
            drafts[b, cut[b]] = (am[b, cut[b]] + 1 + rng.integers(0, V - 1)) % V
            drafts[b, cut[b] + 1:] = rng.integers(-1, V, size=k - cut[b] - 1)
    r = oracle.verify_greedy(logits, drafts.astype(np.int32))
    matches = drafts == am[:, :k]
    correct_len = np.cumprod(matches, axis=1).sum(axis=1)
    assert np.array_equal(r["accept_len"], correct_len)
    assert np.array_equal(correct_len, cut)
    bonus = am[np.arange(B), correct_len]
    for b in range(B):
        j = correct_len[b]
        assert list(r["out_tokens"][b, :j]) == list(drafts[b, :j])
        assert r["out_tokens"][b, j] == bonus[b]
        assert (r["out_tokens"][b, j + 1:] == -1).all()


def test_greedy_invalid_draft_stops(oracle):
    logits = np.zeros((1, 3, 4))
    logits[0, :, 2] = 1.0
    r = oracle.verify_greedy(logits, np.array([[2, -1]], np.int32))
    assert r["accept_len"][0] == 1 and list(r["out_tokens"][0]) == [2, 2, -1]


# --------------------------------------------------------------------------------------------
# One round emits 1 to k+1 tokens ("投机解码", opening conclusions and flowchart).
# --------------------------------------------------------------------------------------------
def _qmix(rng, p, alpha):
    """q = lam*p + (1-lam)*d with sum(min(p, q)) = alpha exactly, d ~ Dirichlet(0.1)."""
    while True:
        d = rng.dirichlet(np.full(p.shape[-1], 0.1))
        m = np.minimum(p, d).sum()
        if m < alpha:
            lam = (alpha - m) / (1 - m)
            return lam * p + (1 - lam) * d


def test_tokens_per_round(oracle):
    rng = np.random.default_rng(2)
    B, k, V = 200, 4, 30
    logits = rng.standard_normal((B, k + 1, V)) * 2
    p = special.softmax(logits, axis=-1)
    q = np.stack([[_qmix(rng, p[b, i], 0.6) for i in range(k)] for b in range(B)]).astype(np.float32)
    drafts = np.array([[rng.choice(V, p=q[b, i] / q[b, i].sum()) for i in range(k)] for b in range(B)], np.int32)
    for qq in (q, None):
        r = oracle.verify_rejection(logits, drafts, qq, 1.0, 99, 0)
        assert (r["status"] == 0).all()
        for b in range(B):
            j = r["accept_len"][b]
            assert 0 <= j <= k
            assert list(r["out_tokens"][b, :j]) == list(drafts[b, :j])
            assert 0 <= r["out_tokens"][b, j] < V
            assert (r["out_tokens"][b, j + 1:] == -1).all()


# --------------------------------------------------------------------------------------------
# E(alpha, k) = (1 - alpha^(k+1)) / (1 - alpha): 2.533 at alpha = 0.7, k = 3
# ("投机解码", 一轮出几个 token; "The speculative decoding zoo").  Inputs are built so that
# every position has sum(min(p, q)) = alpha exactly.
# --------------------------------------------------------------------------------------------
def test_expected_tokens_closed_form(oracle):
    rng = np.random.default_rng(20261031)
    alpha, k, V, B = 0.7, 3, 16, 30000
    assert abs((1 - alpha ** (k + 1)) / (1 - alpha) - 2.533) < 1e-3
    p = rng.dirichlet(np.ones(V), size=(B, k + 1))
    q = np.empty((B, k, V))
    for b in range(B):
        for i in range(k):
            q[b, i] = _qmix(rng, p[b, i], alpha)
    cq = np.cumsum(q, axis=-1)
    drafts = (cq < rng.random((B, k, 1)) * cq[..., -1:]).sum(axis=-1).astype(np.int32)
    logits = np.log(p)
    emitted = []
    for offset in range(4):
        r = oracle.verify_rejection(logits, drafts, q.astype(np.float32), 1.0, 7, offset)
        emitted.append(r["accept_len"] + 1)
    emitted = np.concatenate(emitted).astype(np.float64)
    E = (1 - alpha ** (k + 1)) / (1 - alpha)
    se = emitted.std() / np.sqrt(emitted.size)
    # q is rounded to fp32, so alpha is exact only to ~1e-7; far below the statistical error.
    assert abs(emitted.mean() - E) < 4 * se, (emitted.mean(), E, se)
    # The accept length is geometric: P(len = j) = alpha^j (1 - alpha), P(len = k) = alpha^k.
    counts = np.bincount((emitted - 1).astype(int), minlength=k + 1)
    probs = np.array([alpha ** j * (1 - alpha) for j in range(k)] + [alpha ** k])
    assert stats.chisquare(counts, probs * counts.sum()).pvalue > 1e-4


# --------------------------------------------------------------------------------------------
# Multi-position joint distribution: a 4-token Markov target and draft, 2 drafts per round,
# sequences of length 3 compared with the exact joint over 64 outcomes ("投机解码", 数学验证;
# the chain's values are ours, the page does not print them).
# --------------------------------------------------------------------------------------------
def test_markov_joint_distribution(oracle):
    Pm = np.array([[0.50, 0.20, 0.20, 0.10],
                   [0.10, 0.60, 0.10, 0.20],
                   [0.25, 0.25, 0.25, 0.25],
                   [0.05, 0.15, 0.30, 0.50]])
    Qm = np.array([[0.30, 0.30, 0.20, 0.20],
                   [0.40, 0.20, 0.20, 0.20],
                   [0.10, 0.10, 0.70, 0.10],
                   [0.25, 0.25, 0.25, 0.25]])
    n, k, start = 60000, 2, 0
    rng = np.random.default_rng(20261031)
    seqs = [[] for _ in range(n)]
    active = np.arange(n)
    rnd = 0
    while active.size:
        last = np.array([seqs[s][-1] if seqs[s] else start for s in active])
        d1 = (np.cumsum(Qm[last], 1) < rng.random((active.size, 1))).sum(1)
        d2 = (np.cumsum(Qm[d1], 1) < rng.random((active.size, 1))).sum(1)
        drafts = np.stack([d1, d2], 1).astype(np.int32)
        logits = np.log(np.stack([Pm[last], Pm[d1], Pm[d2]], 1))
        q = np.stack([Qm[last], Qm[d1]], 1).astype(np.float32)
        r = oracle.verify_rejection(logits, drafts, q, 1.0, 7, rnd, req_ids=None)
        for i, s in enumerate(active):
            j = r["accept_len"][i]
            seqs[s].extend(int(t) for t in r["out_tokens"][i, : j + 1])
        active = np.array([s for s in active if len(seqs[s]) < 3], dtype=np.int64)
        rnd += 1
    counts = np.zeros(64)
    for s in seqs:
        a, b, c = s[:3]
        counts[16 * a + 4 * b + c] += 1
    exact = np.array([Pm[start, a] * Pm[a, b] * Pm[b, c]
                      for a in range(4) for b in range(4) for c in range(4)])
    assert stats.chisquare(counts, exact * n).pvalue > 1e-4
    # The same drafts judged with q replaced by one-hot drafts must also keep the joint.


# --------------------------------------------------------------------------------------------
# Trees.
# --------------------------------------------------------------------------------------------
def _chain_tree(drafts_row):
    k = len(drafts_row)
    tokens = np.array([-1] + list(drafts_row), np.int32)
    parents = np.array([-1] + list(range(k)), np.int32)
    return tokens, parents


def test_path_tree_equals_one_hot_chain(oracle):
    # With one child per node the target-only tree rule is the one-hot chain rule
    # ("投机解码": with topk = 1 the tree rule is exactly vLLM's one-hot rule).
    rng = np.random.default_rng(4)
    B, k, V = 400, 5, 12
    logits = (rng.standard_normal((B, k + 1, V)) * 1.5).astype(np.float32)
    am = np.argmax(logits, -1)
    drafts = np.where(rng.random((B, k)) < 0.7, am[:, :k], rng.integers(0, V, (B, k))).astype(np.int32)
    toks, pars = zip(*[_chain_tree(d) for d in drafts])
    toks, pars = np.stack(toks), np.stack(pars)
    for seed in (1, 2):
        c = oracle.verify_rejection(logits, drafts, None, 0.9, seed, 3)
        t = oracle.verify_tree(logits, toks, pars, 1, 0.9, seed, 3)
        assert np.array_equal(c["accept_len"], t["accept_len"])
        assert np.array_equal(c["out_tokens"], t["out_tokens"])
        for b in range(B):
            j = t["accept_len"][b]
            assert list(t["accept_index"][b, : j + 1]) == list(range(j + 1))
    g = oracle.verify_greedy(logits, drafts)
    tg = oracle.verify_tree(logits, toks, pars, 0, 1.0, 0, 0)
    assert np.array_equal(g["accept_len"], tg["accept_len"])
    assert np.array_equal(g["out_tokens"], tg["out_tokens"])


def test_two_level_tree_joint(oracle):
    # Root children {0, 2}; node 1 (token 0) has children {1, 3}; node 2 (token 2) has child {3}.
    # The first two emitted tokens must follow p_root then p_(accepted node); when the first
    # token is not a node, the round stops after it.
    V = 4
    p_root = np.array([0.3, 0.2, 0.4, 0.1])
    p_n1 = np.array([0.1, 0.5, 0.2, 0.2])
    p_n2 = np.array([0.25, 0.25, 0.1, 0.4])
    leaf = np.array([0.25, 0.25, 0.25, 0.25])
    tokens = np.array([-1, 0, 2, 1, 3, 3], np.int32)
    parents = np.array([-1, 0, 0, 1, 1, 2], np.int32)
    rows = np.stack([p_root, p_n1, p_n2, leaf, leaf, leaf])
    n = 200000
    logits = np.broadcast_to(np.log(rows), (n, 6, V)).copy()
    r = oracle.verify_tree(logits, np.broadcast_to(tokens, (n, 6)), np.broadcast_to(parents, (n, 6)),
                           1, 1.0, 20261031, 0)
    first = r["out_tokens"][:, 0]
    assert stats.chisquare(np.bincount(first, minlength=V), p_root * n).pvalue > 1e-4
    for tok, node_row in ((0, p_n1), (2, p_n2)):
        sel = first == tok
        second = r["out_tokens"][sel, 1]
        assert (second >= 0).all()
        assert stats.chisquare(np.bincount(second, minlength=V), node_row * sel.sum()).pvalue > 1e-4
    for tok in (1, 3):
        assert (r["out_tokens"][first == tok, 1] == -1).all()
    # Acceptance at the root is p_root(0) + p_root(2) = 0.7.
    assert abs((r["accept_len"] >= 1).mean() - 0.7) < 4 * np.sqrt(0.21 / n)


def test_tree_structure_checks(oracle):
    V = 10
    ok_t = [-1, 3, 4, 5]
    assert oracle.tree_check(ok_t, [-1, 0, 0, 1], V, 1) == 0
    assert oracle.tree_check(ok_t, [0, 0, 0, 1], V, 1) == 3  # root with a parent
    assert oracle.tree_check(ok_t, [-1, 0, 2, 1], V, 1) == 3  # forward parent
    assert oracle.tree_check(ok_t, [-1, 0, -1, 1], V, 1) == 3  # orphan
    assert oracle.tree_check([-1, 3, 10, 5], [-1, 0, 0, 1], V, 1) == 1
    assert oracle.tree_check([-1, 3, 3, 5], [-1, 0, 0, 1], V, 1) == 4  # duplicate siblings
    assert oracle.tree_check([-1, 3, 3, 5], [-1, 0, 0, 1], V, 0) == 0  # fine when greedy
    assert oracle.tree_check([-1, 3, 3, 3], [-1, 0, 1, 2], V, 1) == 0  # same token, not siblings
    assert oracle.tree_check([-1, -1, -1, 5], [-1, 0, 0, 1], V, 1) == 0  # absent nodes


def test_tree_greedy_follows_argmax(oracle):
    V = 6
    rows = np.full((4, V), -1.0)
    rows[0, 4] = 2.0  # root argmax 4 -> node 2
    rows[2, 1] = 2.0  # node 2 argmax 1 -> node 3
    rows[3, 5] = 2.0  # node 3 is a leaf: bonus 5
    tokens = np.array([-1, 3, 4, 1], np.int32)
    parents = np.array([-1, 0, 0, 2], np.int32)
    r = oracle.verify_tree(rows[None], tokens[None], parents[None], 0, 1.0, 0, 0)
    assert r["accept_len"][0] == 2
    assert list(r["accept_index"][0]) == [0, 2, 3, -1]
    assert list(r["out_tokens"][0]) == [4, 1, 5, -1]
