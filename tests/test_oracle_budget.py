"""Pins of the oracle's adaptive verification budget: the worked example the pages print (budgets
112 / 57 / 7 and their throughputs), brute force over every prefix-closed admission on tiny
inputs, and the tie and range rules.

Planting each of these mistakes in a copy of the oracle fails at least one pin: later positions
first on equal survivals, the higher request first on equal survivals, the last maximum for the
first, the rate without B, cost[b - 1] for cost[b], confidences not multiplied along the drafts,
num_drafts ignored, confidences not clamped to [0, 1], the slots taken worst first."""
import itertools
import json
import os

import numpy as np
import pytest
import torch


def _toy(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "adaptive_budget_toy.json")))
    cm = g["cost_model"]

    def step(tokens):
        return max(cm["weight_bytes"] / cm["bandwidth"], tokens * cm["flop_per_token"] / cm["flops"])

    return g, step, cm["draft_seconds"]


def test_printed_toy_budgets(oracle, golden_dir):
    g, step, t_draft = _toy(golden_dir)
    K = g["inputs"]["K"]
    gen = torch.Generator().manual_seed(0)
    for batch in g["inputs"]["batches"]:
        half = batch // 2
        base = torch.cat([torch.full((half, K), 0.9), torch.full((batch - half, K), 0.55)])
        conf = (base * (torch.rand(batch, K, generator=gen) * 0.2 + 0.9)).clamp(max=0.99).numpy()
        cost = np.array([t_draft + step(batch + b) for b in range(batch * K + 1)])
        r = oracle.plan_budget(conf, cost)
        want = g["printed"][str(batch)]
        assert r["budget"] == want["budget"]
        assert round(r["rate"]) == want["adaptive_tokens_per_s"]
        assert round(float(r["admitted"][:half].mean()), 1) == want["accurate_mean_admitted"]
        assert round(float(r["admitted"][half:].mean()), 1) == want["inaccurate_mean_admitted"]
        assert r["admitted"].sum() == r["budget"]


def test_brute_force_over_prefix_admissions(oracle):
    """For every admission (a_1..a_B), 0 <= a_r <= K, the expected accepted tokens are the sum of
    the admitted survivals; the planner's rate must equal the best rate over all of them."""
    rng = np.random.default_rng(0)
    for trial in range(40):
        B, K = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        conf = rng.random((B, K)).astype(np.float32)
        if trial % 4 == 0:
            conf[rng.random((B, K)) < 0.3] = 1.0
        cost = 1.0 + rng.random(B * K + 1) * 0.5 + np.arange(B * K + 1) * rng.random() * 0.3
        surv = np.cumprod(conf.astype(np.float64), axis=1)
        best = -1.0
        for a in itertools.product(range(K + 1), repeat=B):
            gain = sum(surv[r, : a[r]].sum() for r in range(B))
            best = max(best, (B + gain) / cost[sum(a)])
        r = oracle.plan_budget(conf, cost)
        assert r["rate"] == pytest.approx(best, rel=1e-6)
        assert r["admitted"].sum() == r["budget"]


def test_ties_prefer_earlier_positions_and_ragged_requests(oracle):
    conf = np.array([[1.0, 1.0, 0.5], [1.0, 0.5, 0.5]], np.float32)
    flat = np.ones(7)
    r = oracle.plan_budget(conf, flat * 1.0)  # constant cost: admit every positive slot
    assert r["budget"] == 6 and r["admitted"].tolist() == [3, 3]
    # Survivals: request 0 [1, 1, .5], request 1 [1, .5, .25].  The three slots of survival 1 go
    # first, position 0 of both requests before position 1 of request 0; a fourth slot (.5)
    # costs 0.3 more, so (2 + 3) / 1 = 5 beats (2 + 3.5) / 1.3.
    cost = 1.0 + 0.3 * np.maximum(np.arange(7) - 3, 0)
    r = oracle.plan_budget(conf, cost)
    assert r["budget"] == 3 and r["admitted"].tolist() == [2, 1]
    # Equal survivals at positions 0 and 1 of one request: the earlier position is admitted.
    r = oracle.plan_budget(np.array([[1.0, 1.0]], np.float32), np.array([1.0, 0.5, 10.0]))
    assert r["budget"] == 1 and r["admitted"].tolist() == [1]
    r = oracle.plan_budget(conf, flat, num_drafts=[1, 0])
    assert r["admitted"].tolist() == [1, 0]
    # NaN confidences read as 0; values above 1 as 1.
    r = oracle.plan_budget(np.array([[np.nan, 2.0]], np.float32), np.ones(3))
    assert r["admitted"].tolist() == [0]
    r = oracle.plan_budget(np.array([[2.0, 0.5]], np.float32), np.array([1.0, 1.0, 1.0]))
    assert r["admitted"].tolist() == [2]
    # The clamp decides: read as 1, the survivals [1, .5] make budget 1 best (2 / 1 against
    # 2.5 / 1.3); unclamped, [2, 1] would make it budget 2 (4 / 1.3 against 3 / 1).
    r = oracle.plan_budget(np.array([[2.0, 0.5]], np.float32), np.array([1.0, 1.0, 1.3]))
    assert r["budget"] == 1 and r["admitted"].tolist() == [1] and r["rate"] == pytest.approx(2.0)
    # Equal survivals at the same position of two requests: the lower request is admitted first.
    r = oracle.plan_budget(np.array([[0.5], [0.5]], np.float32), np.array([1.0, 0.5, 10.0]))
    assert r["budget"] == 1 and r["admitted"].tolist() == [1, 0]


def test_zero_gain_keeps_the_smaller_budget(oracle):
    conf = np.array([[0.8, 0.0, 0.0], [0.0, 0.0, 0.0]], np.float32)
    r = oracle.plan_budget(conf, np.ones(7))
    assert r["budget"] == 1 and r["admitted"].tolist() == [1, 0]
