"""Parity of top-k / top-p on the target distribution (spec_verify_rejection_ex /
spec_verify_tree_ex with top_k and top_p, through the C ABI) with the oracle.  bf16 logits hold
many equal values, so ties at the top-k and top-p boundaries are exercised throughout."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_verify_gb300 as sv
from speculative_decoding_verification_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
PROB_RTOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_verify_gb300 import _build

    _build.build()
    oracle.build()
    torch.cuda.set_device(DEV)


def _np(t):
    return t.detach().cpu().numpy()


def _filters(B, V, seed):
    rng = np.random.default_rng(seed)
    tk = rng.choice([0, 1, 3, 20, 400, V - 1, V + 5], B).astype(np.int32)
    tp = rng.choice([1.0, 0.95, 0.8, 0.5, 0.2, 0.05], B).astype(np.float32)
    return tk, tp


def run_chain(inp, tk, tp, with_q=False, temps=None, T=1.0, offset=0):
    B, k, V = inp.shape
    q = inp.q if with_q else None
    dev = lambda a: None if a is None else torch.from_numpy(a).to(DEV)  # noqa: E731
    op = torch.full((B, k + 1, 3), -7.0, device=DEV)
    r = sv.spec_verify_rejection_ex(inp.logits, inp.drafts, q, temperatures=dev(temps), temperature=T,
                                    top_k=dev(tk), top_p=dev(tp), seed=inp.seed, offset=offset, out_probs=op)
    temps_ref = np.full(B, T) if temps is None else temps.astype(np.float64)
    ref = oracle.verify_ex(wl.to_numpy_logits(inp.logits), _np(inp.drafts), None if q is None else _np(q),
                           temps_ref, inp.seed, offset, top_k=tk, top_p=None if tp is None else tp.astype(np.float64))
    torch.cuda.synchronize()
    _compare(_np(r.out_tokens), _np(r.accept_len), ref)
    assert int(_np(r.dev_status)[0]) == int(ref["status"].max())
    got = _np(op).astype(np.float64)
    for b in np.flatnonzero(~ref["boundary"].astype(bool)):
        r = ref["out_probs"][b]
        big = np.abs(r) > 1e-30
        rel = np.abs(got[b][big] - r[big]) / np.abs(r[big])
        assert rel.size == 0 or rel.max() < PROB_RTOL, (b, rel.max())
        assert np.all(np.abs(got[b][~big]) < 1e-29)
    return ref


def _compare(tokens, alen, ref, extra=()):
    """Every request must match, except flagged ones (a top-p crossing within 1e-6 of its mass from
    a value level's edge, or a uniform within 1e-6 of a decision), which must stay rare."""
    flagged = ref["boundary"].astype(bool)
    differ = (tokens != ref["out_tokens"]).any(1) | (alen != ref["accept_len"])
    for g, key in extra:
        differ |= (g != ref[key]).any(1)
    assert not (differ & ~flagged).any(), f"unflagged mismatches at {np.flatnonzero(differ & ~flagged)}"
    assert flagged.sum() <= max(2, len(alen) // 100), f"{flagged.sum()} of {len(alen)} requests flagged"


@pytest.mark.parametrize("V", [1031, 9001, 128256])
def test_topkp_one_hot_chain(V):
    B = 24 if V < 100000 else 8
    inp = wl.chain_sweep(DEV, B=B, k=4, V=V, alpha=0.7)
    tk, tp = _filters(B, V, V)
    one_hot = wl.ChainInputs("one-hot", inp.logits, inp.drafts, None, 1.0, inp.seed)
    run_chain(one_hot, tk, tp)
    run_chain(one_hot, tk, None)
    run_chain(one_hot, None, tp, offset=3)


@pytest.mark.parametrize("V", [4099, 32003])
def test_topkp_with_draft_probs(V):
    inp = wl.chain_sweep(DEV, B=16, k=5, V=V, alpha=0.7)
    tk, tp = _filters(16, V, 7 + V)
    run_chain(inp, tk, tp, with_q=True)


def test_topkp_mixed_temperatures_and_fp32():
    inp = wl.chain_sweep(DEV, B=20, k=3, V=6007, alpha=0.7)
    tk, tp = _filters(20, 6007, 5)
    temps = np.random.default_rng(1).uniform(0.4, 1.5, 20).astype(np.float32)
    temps[::4] = 0.0
    one_hot = wl.ChainInputs("one-hot", inp.logits, inp.drafts, None, 1.0, inp.seed)
    run_chain(one_hot, tk, tp, temps=temps)
    lg32 = inp.logits.float().contiguous()
    run_chain(wl.ChainInputs("fp32", lg32, inp.drafts, None, 1.0, inp.seed), tk, tp, T=0.7)
    run_chain(wl.ChainInputs("fp32", lg32, inp.drafts, inp.q, 1.0, inp.seed), tk, tp, with_q=True, T=1.3)


def test_top_k_one_is_the_argmax_draw():
    """top_k = 1 keeps only the row's maximum value (all tokens sharing it): a draft equal to the
    argmax is always accepted, and the bonus token is the argmax when it is unique."""
    inp = wl.chain_b64k7(DEV, B=16, k=7, V=9001, seed=3)
    tk = np.ones(16, np.int32)
    ref = run_chain(wl.ChainInputs("b", inp.logits, inp.drafts, None, 1.0, inp.seed), tk, None)
    g = oracle.verify_greedy(wl.to_numpy_logits(inp.logits), _np(inp.drafts))
    np.testing.assert_array_equal(ref["accept_len"], g["accept_len"])


def test_topkp_tree():
    tree = wl.tree_b48(DEV, V=8009)
    tk, tp = _filters(48, 8009, 11)
    dev = lambda a: torch.from_numpy(a).to(DEV)  # noqa: E731
    r = sv.spec_verify_tree_ex(tree.logits, tree.node_tokens, tree.parents, top_k=dev(tk), top_p=dev(tp),
                               seed=tree.seed)
    ref = oracle.verify_tree_ex(wl.to_numpy_logits(tree.logits), _np(tree.node_tokens), _np(tree.parents),
                                np.ones(48), tree.seed, 0, top_k=tk, top_p=tp.astype(np.float64))
    torch.cuda.synchronize()
    _compare(_np(r.out_tokens), _np(r.accept_len), ref, extra=[(_np(r.accept_index), "accept_index")])


def test_filters_off_match_the_plain_path():
    inp = wl.chain_b64k7(DEV, B=12, k=7, V=7001, seed=9)
    off_k = torch.zeros(12, dtype=torch.int32, device=DEV)
    off_p = torch.ones(12, dtype=torch.float32, device=DEV)
    a = sv.spec_verify_rejection_ex(inp.logits, inp.drafts, None, top_k=off_k, top_p=off_p, seed=2, offset=1)
    b = sv.spec_verify_rejection(inp.logits, inp.drafts, None, temperature=1.0, seed=2, offset=1)
    torch.cuda.synchronize()
    assert torch.equal(a.out_tokens, b.out_tokens) and torch.equal(a.accept_len, b.accept_len)
