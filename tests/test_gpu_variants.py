"""Parity of the verify variants (spec_verify_rejection_ex / spec_verify_tree_ex, through the C
ABI) with the oracle: relaxed thresholds of target-only decisions and a temperature per request
(greedy and sampled requests in one batch).  Token ids and accept lengths must match exactly,
except for requests the oracle flags as boundary draws."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_verify_gb300 as sv
from speculative_decoding_verification_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_verify_gb300 import _build

    _build.build()
    oracle.build()
    torch.cuda.set_device(DEV)


def _np(t):
    return t.detach().cpu().numpy()


def _temps(B, seed, frac_greedy=0.4):
    rng = np.random.default_rng(seed)
    t = rng.uniform(0.5, 1.6, B).astype(np.float32)
    t[rng.random(B) < frac_greedy] = 0.0
    return t


def run_chain(inp, temps=None, T=1.0, thr=(1.0, 1.0), with_q=False, offset=0, probs=True):
    B, k, V = inp.shape
    q = inp.q if with_q else None
    tt = None if temps is None else torch.from_numpy(temps).to(DEV)
    op = torch.full((B, k + 1, 3), -7.0, device=DEV) if probs else None
    r = sv.spec_verify_rejection_ex(inp.logits, inp.drafts, q, temperatures=tt, temperature=T,
                                    threshold_single=thr[0], threshold_acc=thr[1], seed=inp.seed,
                                    offset=offset, out_probs=op)
    temps_ref = np.full(B, T, np.float64) if temps is None else temps.astype(np.float64)
    ref = oracle.verify_ex(wl.to_numpy_logits(inp.logits), _np(inp.drafts), None if q is None else _np(q),
                           temps_ref, inp.seed, offset, thr[0], thr[1])
    torch.cuda.synchronize()
    ok = ~ref["boundary"].astype(bool)
    np.testing.assert_array_equal(_np(r.accept_len)[ok], ref["accept_len"][ok])
    np.testing.assert_array_equal(_np(r.out_tokens)[ok], ref["out_tokens"][ok])
    assert (~ok).sum() <= max(2, B // 50)
    assert int(_np(r.dev_status)[0]) == int(ref["status"].max())
    if probs:
        got = _np(op)
        for b in np.flatnonzero(ok):
            if temps_ref[b] == 0.0:
                assert not got[b].any()
            else:
                np.testing.assert_allclose(got[b], ref["out_probs"][b], rtol=1e-5, atol=1e-7)
    return r, ref


@pytest.mark.parametrize("thr", [(0.5, 0.5), (1.0, 0.6), (0.3, 1.0)])
def test_relaxed_thresholds_one_hot_chain(thr):
    inp = wl.chain_b64k7(DEV, B=24, k=7, V=9001, seed=11)
    r, ref = run_chain(inp, thr=thr)
    # The relaxed rule accepts at least as much as the exact one on the same uniforms.
    exact = oracle.verify_ex(wl.to_numpy_logits(inp.logits), _np(inp.drafts), None, np.ones(24), inp.seed, 0)
    assert (ref["accept_len"] >= exact["accept_len"]).all()
    assert ref["accept_len"].sum() > exact["accept_len"].sum()


def test_thresholds_of_one_match_the_plain_entry_point():
    inp = wl.chain_sweep(DEV, B=16, k=5, V=12007, alpha=0.7)
    a = sv.spec_verify_rejection_ex(inp.logits, inp.drafts, inp.q, temperature=inp.temperature, seed=3, offset=2)
    b = sv.spec_verify_rejection(inp.logits, inp.drafts, inp.q, temperature=inp.temperature, seed=3, offset=2)
    torch.cuda.synchronize()
    assert torch.equal(a.out_tokens, b.out_tokens) and torch.equal(a.accept_len, b.accept_len)


@pytest.mark.parametrize("with_q", [False, True])
@pytest.mark.parametrize("V", [9001, 128256])
def test_mixed_temperatures_chain(with_q, V):
    B = 24 if V < 100000 else 12
    inp = wl.chain_sweep(DEV, B=B, k=5, V=V, alpha=0.7)
    temps = _temps(B, V)
    temps[0], temps[1] = 0.0, 1.0
    run_chain(inp, temps=temps, with_q=with_q)
    run_chain(inp, temps=temps, with_q=with_q, offset=5)


def test_mixed_relaxed_one_hot_fp32():
    inp = wl.chain_b64k7(DEV, B=20, k=6, V=5003, seed=21)
    lg = inp.logits.float().contiguous()
    inp32 = wl.ChainInputs("fp32", lg, inp.drafts, None, 1.0, inp.seed)
    run_chain(inp32, temps=_temps(20, 5), thr=(0.6, 0.8))


def test_all_greedy_forms():
    inp = wl.chain_b64k7(DEV, B=16, k=7, V=7001, seed=8)
    zeros = np.zeros(16, np.float32)
    r1, _ = run_chain(inp, temps=zeros)
    r2, _ = run_chain(inp, T=0.0)
    g = sv.spec_verify_greedy(inp.logits, inp.drafts)
    torch.cuda.synchronize()
    assert torch.equal(r1.out_tokens, g.out_tokens) and torch.equal(r2.out_tokens, g.out_tokens)


def run_tree(tree, temps=None, T=1.0, thr=(1.0, 1.0)):
    B, N, V = tree.shape
    tt = None if temps is None else torch.from_numpy(temps).to(DEV)
    r = sv.spec_verify_tree_ex(tree.logits, tree.node_tokens, tree.parents, temperatures=tt, temperature=T,
                               threshold_single=thr[0], threshold_acc=thr[1], seed=tree.seed)
    temps_ref = np.full(B, T, np.float64) if temps is None else temps.astype(np.float64)
    ref = oracle.verify_tree_ex(wl.to_numpy_logits(tree.logits), _np(tree.node_tokens), _np(tree.parents),
                                temps_ref, tree.seed, 0, thr[0], thr[1])
    torch.cuda.synchronize()
    ok = ~ref["boundary"].astype(bool)
    np.testing.assert_array_equal(_np(r.accept_len)[ok], ref["accept_len"][ok])
    np.testing.assert_array_equal(_np(r.out_tokens)[ok], ref["out_tokens"][ok])
    np.testing.assert_array_equal(_np(r.accept_index)[ok], ref["accept_index"][ok])
    assert (~ok).sum() <= 2
    assert int(_np(r.dev_status)[0]) == int(ref["status"].max())
    return ref


@pytest.mark.parametrize("thr", [(1.0, 1.0), (0.5, 0.5), (0.4, 0.9)])
def test_tree_relaxed_and_mixed(thr):
    tree = wl.tree_b48(DEV, V=6007)
    ref = run_tree(tree, thr=thr)
    run_tree(tree, temps=_temps(48, 17), thr=thr)
    if thr != (1.0, 1.0):
        exact = run_tree(tree)
        assert ref["accept_len"].sum() >= exact["accept_len"].sum()


def test_tree_all_greedy_matches_mode_0():
    tree = wl.tree_b48(DEV, B=12, V=6007)
    r = sv.spec_verify_tree_ex(tree.logits, tree.node_tokens, tree.parents, temperature=0.0)
    g = sv.spec_verify_tree(tree.logits, tree.node_tokens, tree.parents, mode=0)
    torch.cuda.synchronize()
    assert torch.equal(r.out_tokens, g.out_tokens) and torch.equal(r.accept_index, g.accept_index)


def test_full_size_mixed_sampled():
    """The b64k7 workload with a temperature per request: a sample of requests."""
    inp = wl.chain_b64k7(DEV)
    temps = _temps(64, 99)
    tt = torch.from_numpy(temps).to(DEV)
    r = sv.spec_verify_rejection_ex(inp.logits, inp.drafts, None, temperatures=tt, seed=inp.seed, offset=1)
    ids = np.array([0, 3, 17, 31, 40, 63], np.int32)
    ref = oracle.verify_ex(wl.to_numpy_logits(inp.logits), _np(inp.drafts), None, temps.astype(np.float64),
                           inp.seed, 1, req_ids=ids)
    torch.cuda.synchronize()
    ok = ~ref["boundary"].astype(bool)
    np.testing.assert_array_equal(_np(r.out_tokens)[ids][ok], ref["out_tokens"][ok])
    np.testing.assert_array_equal(_np(r.accept_len)[ids][ok], ref["accept_len"][ok])


def test_invalid_options():
    inp = wl.chain_tiny(DEV)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_rejection_ex(inp.logits, inp.drafts, inp.q, threshold_acc=0.5)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_rejection_ex(inp.logits, inp.drafts, None, threshold_single=1.5)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_rejection_ex(inp.logits, inp.drafts, None, temperature=-1.0)
