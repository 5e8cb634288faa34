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


# Edges of the one-read threshold kernel (bf16 rows with top-k <= 256 and at most 32768 vectors):
# every case is compared with the oracle, and no stage wait may run out.

@pytest.mark.parametrize("shift", [1, 3, 6])
def test_topkp_unaligned_rows(shift):
    """A logits base off the 16-byte grid: every row has a head and a tail outside its aligned
    body, read element by element and folded into the first group."""
    base = wl.chain_sweep(DEV, B=6, k=3, V=10007, alpha=0.7)
    B, k, V = base.logits.shape[0], 3, 10007
    buf = torch.empty(B * (k + 1) * V + 8, dtype=torch.bfloat16, device=DEV)
    view = buf[shift:shift + B * (k + 1) * V].view(B, k + 1, V)
    view.copy_(base.logits)
    tk = np.array([1, 7, 50, 200, 512, 3], np.int32)
    tp = np.array([1.0, 0.9, 0.5, 0.95, 1.0, 0.2], np.float32)
    one_hot = wl.ChainInputs("unaligned", view, base.drafts, None, 1.0, base.seed)
    run_chain(one_hot, tk, tp, offset=shift)
    run_chain(one_hot, tk, None, offset=shift)


def test_topkp_k_at_the_ring_limit():
    """top-k 256 (the one-read kernel's largest) and 257, 512 (the general kernel) on the same rows."""
    inp = wl.chain_sweep(DEV, B=4, k=3, V=32000, alpha=0.7)
    one_hot = wl.ChainInputs("one-hot", inp.logits, inp.drafts, None, 1.0, inp.seed)
    for kk in (256, 257, 512):
        tk = np.full(4, kk, np.int32)
        run_chain(one_hot, tk, np.array([1.0, 0.9, 0.99, 0.6], np.float32))


@pytest.mark.parametrize("V", [262144, 262160])
def test_topkp_longest_rows(V):
    """Rows of exactly 32768 vectors (the one-read kernel's limit) and just above it (general)."""
    inp = wl.chain_sweep(DEV, B=2, k=1, V=V, alpha=0.7)
    one_hot = wl.ChainInputs("one-hot", inp.logits, inp.drafts, None, 1.0, inp.seed)
    run_chain(one_hot, np.array([50, 300], np.int32), np.array([0.9, 1.0], np.float32))


@pytest.mark.parametrize("V", [5, 9, 17, 40])
def test_topkp_tiny_rows(V):
    """Rows with no or few aligned vectors: the head and tail elements carry the row."""
    inp = wl.chain_sweep(DEV, B=6, k=2, V=V, alpha=0.7)
    one_hot = wl.ChainInputs("one-hot", inp.logits, inp.drafts, None, 1.0, inp.seed)
    tk = np.array([1, 2, 3, V - 1, 4, 2], np.int32)
    run_chain(one_hot, tk, np.array([1.0, 0.5, 0.9, 0.99, 1.0, 0.3], np.float32))


def test_topkp_heavy_ties_and_signed_zeros():
    """Logits on a coarse grid (few value levels, long ties at every boundary) with zeros of both
    signs, including rows whose maximum is zero."""
    B, k, V = 8, 3, 20011
    g = torch.Generator(device=DEV).manual_seed(21)
    lv = torch.randint(-6, 3, (B, k + 1, V), generator=g, device=DEV).float() * 0.5
    lv[:, :, ::3] = torch.where(lv[:, :, ::3] == 0, -0.0, lv[:, :, ::3])
    lv[:4] = torch.minimum(lv[:4], torch.zeros_like(lv[:4]))  # rows topped by +0 / -0
    lv[:4, :, ::5] = -0.0
    logits = lv.to(torch.bfloat16).contiguous()
    drafts = torch.randint(0, V, (B, k), generator=g, device=DEV, dtype=torch.int32)
    inp = wl.ChainInputs("ties", logits, drafts, None, 1.0, 77)
    tk = np.array([1, 5, 100, 512, 30, 2, 256, 9], np.int32)
    tp = np.array([0.9, 0.5, 1.0, 0.8, 0.3, 1.0, 0.99, 0.6], np.float32)
    run_chain(inp, tk, tp)
    run_chain(inp, tk, None, offset=4)


def test_no_wait_ran_out():
    inp = wl.chain_b64k7(DEV, B=16, k=7, V=128256, seed=4)
    tk = torch.full((16,), 50, dtype=torch.int32, device=DEV)
    tp = torch.full((16,), 0.9, dtype=torch.float32, device=DEV)
    sv.spec_verify_wait_timeouts()
    for i in range(3):
        sv.spec_verify_rejection_ex(inp.logits, inp.drafts, None, top_k=tk, top_p=tp, seed=1, offset=i)
    torch.cuda.synchronize()
    assert sv.spec_verify_wait_timeouts() == 0


def test_topkp_ring_hands_rows_to_the_general_kernel():
    """One call whose rows take every route: ordinary rows (the one-read kernel), fully tied rows
    (more groups reach L than the kernel lists, so the general kernel takes them), rows with one
    logit far above the rest (the key range [L, max] is too wide), and top-p alone (general)."""
    B, k, V = 6, 3, 128256
    g = torch.Generator(device=DEV).manual_seed(31)
    lv = torch.randn((B, k + 1, V), generator=g, device=DEV) * 2.0
    lv[1] = 0.75                      # every logit equal
    lv[2] = torch.randn((k + 1, V), generator=g, device=DEV) * 0.5
    lv[2, :, 777] = 90.0              # one spike far above a flat row
    lv[3, :, ::2] = 1.5               # half the row tied at one level
    logits = lv.to(torch.bfloat16).contiguous()
    drafts = torch.randint(0, V, (B, k), generator=g, device=DEV, dtype=torch.int32)
    drafts[2, 0] = 777
    inp = wl.ChainInputs("routes", logits, drafts, None, 1.0, 91)
    tk = np.array([50, 20, 100, 200, 0, 256], np.int32)
    tp = np.array([0.9, 1.0, 0.95, 0.5, 0.8, 1.0], np.float32)
    run_chain(inp, tk, tp)
    run_chain(inp, tk, None, offset=2)
    assert sv.spec_verify_wait_timeouts() == 0
