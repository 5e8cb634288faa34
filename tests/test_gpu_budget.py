"""Parity of the GPU adaptive verification budget (spec_verify_plan_budget, through the C ABI)
with the oracle: the budget and every request's admitted count must match exactly, except where
the oracle flags another budget within 1e-12 of the best rate."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_verify_gb300 as sv

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_verify_gb300 import _build

    _build.build()
    torch.cuda.set_device(DEV)


def run(conf, cost, num_drafts=None):
    c = torch.from_numpy(np.ascontiguousarray(conf, np.float32)).to(DEV)
    k = torch.from_numpy(np.ascontiguousarray(cost, np.float64)).to(DEV)
    nd = None if num_drafts is None else torch.from_numpy(np.asarray(num_drafts, np.int32)).to(DEV)
    adm, bud, rate = sv.spec_verify_plan_budget(c, k, nd)
    ref = oracle.plan_budget(conf, cost, num_drafts)
    torch.cuda.synchronize()
    if not ref["boundary"]:
        assert int(bud.item()) == ref["budget"]
        np.testing.assert_array_equal(adm.cpu().numpy(), ref["admitted"])
        assert float(rate.item()) == pytest.approx(ref["rate"], rel=1e-12)
    return ref


def _cost(B, K, rng, kind):
    b = np.arange(B * K + 1)
    if kind == "roofline":  # memory floor, then linear in tokens
        return 1e-3 + 0.25e-3 + np.maximum(0.0, (B + b) * 3e-5 - 1e-3)
    if kind == "steps":  # padded to captured sizes: a step function
        return 1.0 + np.ceil((B + b) / 64.0) * 0.05
    return 1.0 + rng.random(B * K + 1)


@pytest.mark.parametrize("B,K", [(1, 1), (3, 5), (16, 7), (128, 7), (512, 7), (250, 63), (2048, 8), (16384, 1)])
@pytest.mark.parametrize("kind", ["roofline", "steps", "random"])
def test_budget_random(B, K, kind):
    rng = np.random.default_rng(B * 100 + K)
    conf = rng.beta(3, 1, (B, K)).astype(np.float32)
    conf[rng.random((B, K)) < 0.05] = 1.0
    run(conf, _cost(B, K, rng, kind))


def test_budget_ties_ragged_and_odd_values():
    rng = np.random.default_rng(7)
    B, K = 300, 9
    conf = np.round(rng.random((B, K)) * 4) / 4  # many equal survivals
    conf = conf.astype(np.float32)
    conf[0, 0] = np.nan
    conf[1, :] = 2.0
    conf[2, 1] = -0.0
    conf[3, :] = -1.0
    nd = rng.integers(0, K + 1, B)
    nd[4] = -3
    for kind in ("roofline", "steps", "random"):
        run(conf, _cost(B, K, rng, kind), nd)
        run(conf, _cost(B, K, rng, kind))


def test_printed_toy_on_the_gpu():
    g = json.load(open(os.path.join(GOLDEN, "adaptive_budget_toy.json")))
    cm = g["cost_model"]
    K = g["inputs"]["K"]
    gen = torch.Generator().manual_seed(0)
    for batch in g["inputs"]["batches"]:
        half = batch // 2
        base = torch.cat([torch.full((half, K), 0.9), torch.full((batch - half, K), 0.55)])
        conf = (base * (torch.rand(batch, K, generator=gen) * 0.2 + 0.9)).clamp(max=0.99).numpy()
        step = [max(cm["weight_bytes"] / cm["bandwidth"], (batch + b) * cm["flop_per_token"] / cm["flops"])
                for b in range(batch * K + 1)]
        cost = cm["draft_seconds"] + np.array(step)
        ref = run(conf, cost)
        assert ref["budget"] == g["printed"][str(batch)]["budget"]


@pytest.mark.parametrize("B,K", [(2049, 1), (683, 6), (1, 64), (2, 64), (4095, 4)])
def test_budget_slot_counts_across_cta_slices(B, K):
    """Slot counts just past the planner's 2048-slot CTA slices, and the longest drafts."""
    rng = np.random.default_rng(B * 7 + K)
    conf = rng.beta(3, 1, (B, K)).astype(np.float32)
    for kind in ("roofline", "random"):
        run(conf, _cost(B, K, rng, kind))
        run(conf, _cost(B, K, rng, kind), rng.integers(0, K + 1, B))


def test_budget_costs_over_a_wide_exponent_range():
    """Costs from 1e-200 to 1e200: the rates' binary exponents span most of fp64's range."""
    rng = np.random.default_rng(11)
    for B, K in ((64, 7), (700, 5)):
        conf = rng.beta(3, 1, (B, K)).astype(np.float32)
        run(conf, 10.0 ** rng.uniform(-200, 200, B * K + 1))
        run(conf, 10.0 ** rng.uniform(-5, 5, B * K + 1) * 1e-150)


def test_budget_exact_rate_ties_take_the_first_budget():
    """Every budget at exactly the same rate, a power of two, which the planner's rate keys carry
    exactly: the first maximum, budget 0, admitting nothing.  (The oracle flags such calls as
    boundary cases; the rule itself fixes the answer.  Tied rates whose quotient is not exact in
    the keys' arithmetic may come out in either order, as for any two rates within 2^-44.)"""
    for B, K in ((5, 3), (512, 7), (2048, 8)):
        conf = np.ones((B, K), np.float32)  # survivals 1: gain[b] = b exactly
        for scale in (1.0, 4.0, 0.125):
            cost = scale * (B + np.arange(B * K + 1, dtype=np.float64))
            c = torch.from_numpy(conf).to(DEV)
            k = torch.from_numpy(cost).to(DEV)
            adm, bud, rate = sv.spec_verify_plan_budget(c, k, None)
            torch.cuda.synchronize()
            assert int(bud.item()) == 0
            assert not adm.cpu().numpy().any()
            assert float(rate.item()) == pytest.approx(1.0 / scale, rel=1e-12)
