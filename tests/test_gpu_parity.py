"""Parity of the CUDA verifier (through its C ABI) with the CPU oracle.

Token ids and accept lengths must match exactly, except for requests the oracle flags as
boundary draws (a decision within 1e-6 relative of its boundary), which are counted and must
stay rare; probabilities must agree within 1e-5 relative.
"""
import ctypes

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


def _req_sample(B, n, seed=0):
    if B <= n:
        return np.arange(B, dtype=np.int32)
    rng = np.random.default_rng(seed)
    idx = np.sort(rng.choice(B, size=n - 2, replace=False))
    return np.unique(np.concatenate([[0, B - 1], idx])).astype(np.int32)


def _compare(gpu_tokens, gpu_len, ref, ids, extra=None):
    """Exact agreement outside the oracle's boundary draws.  A draw is flagged when its uniform lies
    within 1e-6 of a decision boundary (for a draw, 1e-6 * Z of its token's interval); at
    V = 128256 that is a tenth of an average token's mass, so about one draw in twenty is flagged.
    The GPU decides in fp32, about 1e-7 * Z from the exact boundary, so flagged draws must still
    agree almost always."""
    gt, gl = _np(gpu_tokens)[ids], _np(gpu_len)[ids]
    flagged = ref.get("boundary", np.zeros(len(ids), np.int32)).astype(bool)
    differ = (gl != ref["accept_len"]) | (gt != ref["out_tokens"]).any(1)
    if extra is not None:
        differ |= (_np(extra[0])[ids] != ref[extra[1]]).any(1)
    assert not (differ & ~flagged).any(), f"requests {np.flatnonzero(differ & ~flagged)} differ outside the boundary"
    assert (differ & flagged).sum() <= max(1, len(ids) // 50), f"{(differ & flagged).sum()} flagged requests differ"
    assert flagged.sum() <= max(2, len(ids) // 6), f"{flagged.sum()} of {len(ids)} requests flagged"
    return int(flagged.sum())


def _check_probs(out_probs, ref, ids):
    gp = _np(out_probs)[ids].astype(np.float64)
    rp = ref["out_probs"]
    ok = ~ref["boundary"].astype(bool)
    for col in (0, 1, 2):
        g, r = gp[ok][..., col], rp[ok][..., col]
        big = np.abs(r) > 1e-30
        rel = np.abs(g[big] - r[big]) / np.abs(r[big])
        assert rel.size == 0 or rel.max() < PROB_RTOL, (col, rel.max())
        assert np.all(np.abs(g[~big]) < 1e-29)


def run_chain(inp: wl.ChainInputs, mode: str, offset=0, ids=None, want_probs=True):
    B, k, V = inp.shape
    ids = np.arange(B, dtype=np.int32) if ids is None else ids
    lg = wl.to_numpy_logits(inp.logits)
    d = _np(inp.drafts)
    if mode == "greedy":
        r = sv.spec_verify_greedy(inp.logits, inp.drafts)
        ref = oracle.verify_greedy(lg, d, req_ids=ids)
        _compare(r.out_tokens, r.accept_len, ref, ids)
    else:
        q = inp.q if mode == "standard" else None
        r = sv.spec_verify_rejection(inp.logits, inp.drafts, q, temperature=inp.temperature,
                                     seed=inp.seed, offset=offset, want_probs=want_probs)
        ref = oracle.verify_rejection(lg, d, None if q is None else _np(q), inp.temperature,
                                      inp.seed, offset, req_ids=ids)
        _compare(r.out_tokens, r.accept_len, ref, ids)
        if want_probs:
            _check_probs(r.out_probs, ref, ids)
    torch.cuda.synchronize()
    st = int(_np(r.dev_status)[0])
    assert st == int(ref["status"].max()) or len(ids) < B
    return r, ref


def run_tree(inp: wl.TreeInputs, mode: int, offset=0, ids=None):
    B, N, V = inp.shape
    ids = np.arange(B, dtype=np.int32) if ids is None else ids
    lg = wl.to_numpy_logits(inp.logits)
    r = sv.spec_verify_tree(inp.logits, inp.node_tokens, inp.parents, mode=mode,
                            temperature=inp.temperature, seed=inp.seed, offset=offset)
    ref = oracle.verify_tree(lg, _np(inp.node_tokens), _np(inp.parents), mode, inp.temperature,
                             inp.seed, offset, req_ids=ids)
    _compare(r.out_tokens, r.accept_len, ref, ids, extra=(r.accept_index, "accept_index"))
    torch.cuda.synchronize()
    return r, ref


# --------------------------------------------------------------------------------------------
# RNG
# --------------------------------------------------------------------------------------------
def test_philox_words_match_oracle():
    for seed, offset in ((0, 0), (20261031, 5), (2**64 - 1, 2**63 + 3)):
        words = _np(sv.spec_verify_philox(seed, offset, 9, 301)).view(np.uint32)
        for slot in (0, 4, 8):
            for req in (0, 1, 150, 300):
                ref = oracle.philox4x32_10([slot, req, offset & 0xFFFFFFFF, offset >> 32],
                                           [seed & 0xFFFFFFFF, seed >> 32])
                assert list(words[slot, req]) == list(ref)


# --------------------------------------------------------------------------------------------
# Chain: the tiny fp32 workload in every mode, several offsets
# --------------------------------------------------------------------------------------------
@pytest.mark.parametrize("mode", ["greedy", "standard", "onehot"])
def test_tiny(mode):
    inp = wl.chain_tiny(DEV)
    for off in range(4):
        run_chain(inp, mode, offset=off)


@pytest.mark.parametrize("V", [20000, 20001, 4099, 131])
@pytest.mark.parametrize("mode", ["greedy", "onehot", "standard"])
def test_multi_tile_ragged(mode, V):
    if mode == "standard":
        inp = wl.chain_sweep(DEV, B=12, k=5, V=V, alpha=0.6)
    else:
        inp = wl.chain_b64k7(DEV, B=16, k=7, V=V, seed=99 + V)
    for off in range(3):
        run_chain(inp, mode, offset=off)


@pytest.mark.parametrize("T", [0.3, 0.8, 2.5])
def test_temperatures(T):
    inp = wl.chain_b64k7(DEV, B=8, k=5, V=9000, seed=5, T=T)
    run_chain(inp, "onehot")
    inp = wl.chain_sweep(DEV, B=6, k=3, V=9000, alpha=0.5, T=T)
    run_chain(inp, "standard")


def test_fp32_logits_large_vocab():
    inp = wl.chain_b64k7(DEV, B=6, k=4, V=50001, seed=8, dtype=torch.float32)
    for mode in ("greedy", "onehot"):
        run_chain(inp, mode)


@pytest.mark.parametrize("shift", [1, 3, 5, 7])
def test_unaligned_logits(shift):
    base = wl.chain_b64k7(DEV, B=5, k=3, V=10007, seed=shift)
    B, k, V = base.shape
    buf = torch.empty(B * (k + 1) * V + 8, dtype=torch.bfloat16, device=DEV)
    view = buf[shift:shift + B * (k + 1) * V].view(B, k + 1, V)
    view.copy_(base.logits)
    inp = wl.ChainInputs("unaligned", view, base.drafts, None, 1.0, base.seed)
    for mode in ("greedy", "onehot"):
        run_chain(inp, mode)


def test_many_requests_small_vocab():
    inp = wl.chain_b64k7(DEV, B=512, k=7, V=1024, seed=3)
    for mode in ("greedy", "onehot"):
        run_chain(inp, mode, offset=1)
    inp = wl.chain_sweep(DEV, B=300, k=3, V=1000, alpha=0.35)
    run_chain(inp, "standard")


def test_k0_and_single_request():
    inp = wl.chain_b64k7(DEV, B=3, k=0, V=7777, seed=4)
    r, _ = run_chain(inp, "onehot")
    assert (_np(r.accept_len) == 0).all()
    run_chain(inp, "greedy")
    inp = wl.chain_b64k7(DEV, B=1, k=2, V=300000, seed=6)
    run_chain(inp, "onehot")


def test_absent_drafts():
    inp = wl.chain_b64k7(DEV, B=10, k=6, V=3001, seed=12)
    d = inp.drafts.clone()
    d[0, 0] = -1
    d[1, 3:] = -1
    d[2, 5] = -1
    inp.drafts = d
    for mode in ("greedy", "onehot"):
        r, _ = run_chain(inp, mode)
        assert _np(r.accept_len)[0] == 0
    q_inp = wl.chain_sweep(DEV, B=10, k=6, V=3001, alpha=0.7)
    dq = q_inp.drafts.clone()
    dq[0, 0] = -1
    dq[4, 2:] = -1
    q_inp.drafts = dq
    run_chain(q_inp, "standard")


def test_greedy_ties_lowest_index():
    B, k, V = 20, 4, 3000
    g = torch.Generator(device=DEV).manual_seed(1)
    logits = torch.randint(-3, 4, (B, k + 1, V), generator=g, device=DEV).float().to(torch.bfloat16)
    am = torch.argmax(logits.float(), -1)
    drafts = am[:, :k].int().contiguous()
    inp = wl.ChainInputs("ties", logits.contiguous(), drafts, None, 1.0, 0)
    r, _ = run_chain(inp, "greedy")
    assert (_np(r.accept_len) == k).all()


# --------------------------------------------------------------------------------------------
# Full-size configurations, every request compared with the oracle
# --------------------------------------------------------------------------------------------
def test_full_b64k7_onehot():
    inp = wl.chain_b64k7(DEV)
    for off in (0, 1):
        run_chain(inp, "onehot", offset=off)
    run_chain(inp, "greedy")


def test_full_b1k3_standard():
    inp = wl.chain_b1k3(DEV)
    for off in range(3):
        run_chain(inp, "standard", offset=off)


@pytest.mark.parametrize("mode", [0, 1])
def test_full_tree(mode):
    inp = wl.tree_b48(DEV)
    for off in (0, 1):
        run_tree(inp, mode, offset=off)


def test_sweep_cells_sampled():
    for B, k, alpha in ((8, 3, 0.35), (32, 1, 0.7), (64, 7, 0.7)):
        inp = wl.chain_sweep(DEV, B=B, k=k, alpha=alpha)
        run_chain(inp, "standard", ids=_req_sample(B, 4))


def test_sweep_largest_cell():
    # The sweep's largest cell (B=512, k=7, 1.05 GB of logits and 1.84 GB of q), every request.
    inp = wl.chain_sweep(DEV, B=512, k=7, alpha=0.35)
    run_chain(inp, "standard")


def _stops_at(B, k, V, stops, seed, T=1.0, dtype=torch.bfloat16):
    """A chain whose round stops at row stops[b] of request b (almost surely): logits ~N(0, 3^2);
    on each row before the stop the draft sits on a token raised 40 above the row's maximum
    (accepted with p(x) ~ 1), at the stop row the draft is a uniform token of an untouched row
    (rejected with probability ~1, and the draw there lands anywhere in the row); stops[b] = k
    gives the bonus row.  Drafts after the stop are uniform."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn((B, k + 1, V), generator=g, device=DEV) * 3.0
    drafts = torch.randint(0, V, (B, k), generator=g, device=DEV)
    top = x.max(dim=-1).values
    for b in range(B):
        for i in range(min(int(stops[b]), k)):
            x[b, i, drafts[b, i]] = top[b, i] + 40.0
    return wl.ChainInputs("stops_at", x.to(dtype).contiguous(), drafts.int().contiguous(), None, T, seed)


def test_onehot_stops_at_every_row_large_vocab():
    # V = 128256, k = 7: requests stopping at each row 0..6 and at the bonus row 7, so the stop
    # row's draw (locate + rescan of a 32-record row) runs at every row of the finaliser.
    k, V = 7, 128256
    stops = np.array([0, 1, 2, 3, 4, 5, 6, 7, 3, 7, 0, 5], np.int64)
    inp = _stops_at(len(stops), k, V, stops, 501)
    for off in (0, 1):
        r, ref = run_chain(inp, "onehot", offset=off)
        np.testing.assert_array_equal(ref["accept_len"], stops)


@pytest.mark.parametrize("k", [12, 40])
def test_long_chains_large_vocab(k):
    # Stop rows at and beyond the finaliser's eighth warp (rows loop) on 32-record rows, in every
    # chain mode: one-hot, greedy, block (one-hot and with draft probabilities), standard.
    V = 128256
    stops = np.array([0, 8, 9, k - 1, k, 11 if k > 11 else 3], np.int64)
    inp = _stops_at(len(stops), k, V, stops, 600 + k)
    r, ref = run_chain(inp, "onehot")
    np.testing.assert_array_equal(ref["accept_len"], stops)
    run_chain(inp, "greedy")
    lg, d = wl.to_numpy_logits(inp.logits), _np(inp.drafts)
    b = sv.spec_verify_block(inp.logits, inp.drafts, None, temperature=1.0, seed=inp.seed, offset=0)
    _compare(b.out_tokens, b.accept_len, oracle.verify_block(lg, d, None, 1.0, inp.seed, 0),
             np.arange(len(stops), dtype=np.int32))
    q_inp = wl.chain_sweep(DEV, B=3, k=k, V=V, alpha=0.9)
    run_chain(q_inp, "standard")
    qlg, qd, qq = wl.to_numpy_logits(q_inp.logits), _np(q_inp.drafts), _np(q_inp.q)
    b = sv.spec_verify_block(q_inp.logits, q_inp.drafts, q_inp.q, temperature=1.0, seed=q_inp.seed, offset=0)
    _compare(b.out_tokens, b.accept_len, oracle.verify_block(qlg, qd, qq, 1.0, q_inp.seed, 0),
             np.arange(3, dtype=np.int32))


def _deep_path_tree(B, N, V, topk, steps, seed):
    """A tree_b48-shaped random tree per request whose deepest root-to-leaf path is made
    dominant: on that path each node's token is raised 40 above its parent row's maximum, so the
    target-only and greedy walks follow it to its leaf (the last node on it ends the walk)."""
    t = wl.tree_b48(DEV, B=B, N=N, V=V, topk=topk, steps=steps, seed=seed)
    x = t.logits.float()
    pa = _np(t.parents)
    tok = _np(t.node_tokens)
    top = x.max(dim=-1).values
    for b in range(B):
        depth = np.zeros(N, np.int64)
        for j in range(1, N):
            depth[j] = depth[pa[b, j]] + 1
        leaf = int(np.argmax(depth))
        node = leaf
        while node > 0:
            x[b, pa[b, node], int(tok[b, node])] = top[b, pa[b, node]] + 40.0
            node = int(pa[b, node])
    return wl.TreeInputs("deep_path", x.to(torch.bfloat16).contiguous(), t.node_tokens, t.parents, 1.0, seed + 17)


@pytest.mark.parametrize("N,topk,steps", [(16, 4, 15), (64, 3, 40)])
def test_trees_large_vocab_deep_stops(N, topk, steps):
    # Rows 8 and up are each warp's second row in the finaliser: the walks stop at such nodes.
    inp = _deep_path_tree(4, N, 151936, topk, steps, 700 + N)
    for mode in (0, 1):
        r, ref = run_tree(inp, mode)
        last = ref["accept_index"][np.arange(4), ref["accept_len"]]
        assert int(last.max()) >= 8, (ref["accept_len"], last)


def _dominant_chain(B, k, V, T, seed, hit):
    """Logits ~N(0,1) with a +25 peak per row; the draft of slot i is row i's peak when hit[b, i]
    (accepted with p(x) ~ 1), else a random other token (rejected)."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn((B, k + 1, V), generator=g, device=DEV)
    peak = torch.randint(0, V, (B, k + 1, 1), generator=g, device=DEV)
    x.scatter_add_(2, peak, torch.full((B, k + 1, 1), 25.0, device=DEV))
    other = (peak[:, :k, 0] + 1 + torch.randint(0, V - 1, (B, k), generator=g, device=DEV)) % V
    drafts = torch.where(hit, peak[:, :k, 0], other).to(torch.int32).contiguous()
    return wl.ChainInputs("dominant", x.to(torch.bfloat16).contiguous(), drafts, None, T, seed)


@pytest.mark.parametrize("k", [12, 40, 63])
def test_long_chains(k):
    # More rows than the finaliser has warps (its rows loop) and, past 32 drafts, more than one
    # ballot of draft slots.  Drafts on a +25 peak are accepted, so the runs are long.
    B, V = 6, 3001
    hit = torch.ones((B, k), dtype=torch.bool, device=DEV)
    hit[1, k // 2] = False
    hit[2, k - 1] = False
    hit[3, 5] = False
    inp = _dominant_chain(B, k, V, 1.0, 70 + k, hit)
    r, ref = run_chain(inp, "onehot")
    assert int(ref["accept_len"].max()) >= min(k, 32), ref["accept_len"]
    run_chain(inp, "greedy")
    q_inp = wl.chain_sweep(DEV, B=5, k=k, V=V, alpha=0.8)
    run_chain(q_inp, "standard")


@pytest.mark.parametrize("T", [1.0, 0.05])
def test_dominant_child_low_temperature(T):
    # A draft far above every other token of its row (at T = 0.05 its weight is 2^500 times the
    # rest in the row's own reference): p(x) ~ 1, no overflow, no fault.
    B, k, V = 8, 5, 5000
    g = torch.Generator(device=DEV).manual_seed(9)
    hit = torch.rand((B, k), generator=g, device=DEV) < 0.8
    inp = _dominant_chain(B, k, V, T, 80, hit)
    r, ref = run_chain(inp, "onehot")
    assert int(ref["status"].max()) == 0
    assert int(_np(r.dev_status)[0]) == 0


def test_graph_captured_calls_match_direct_calls():
    # Calls captured in a CUDA graph (the two kernels chained by programmatic dependent launch)
    # give the same tokens as the same calls made directly.
    from speculative_decoding_verification_verify_gb300 import binding

    lib = binding.load_library()
    sets = [wl.chain_b64k7(DEV, B=24, k=7, V=20000, seed=900 + i) for i in range(3)]
    B, k, V = sets[0].shape
    nb = sv.spec_verify_workspace_bytes(sv.MODE_REJECTION, B, k, V)
    ws = torch.zeros(nb, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = [(torch.full((B, k + 1), -7, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV))
            for _ in range(6)]
    P = lambda t: ctypes.c_void_p(t.data_ptr())

    def call(i):
        x = sets[i % 3]
        o, a = outs[i]
        rc = lib.spec_verify_rejection(P(x.logits), sv.BF16, P(x.drafts), None, B, k, V, 1.0, x.seed, 50 + i,
                                       P(o), P(a), None, P(ws), nb, P(st),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0

    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(3, 6):
            call(i)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    # The graph's calls used offsets 53..55; compare with direct calls at those offsets.
    for j, i in enumerate(range(3, 6)):
        x = sets[i % 3]
        d = sv.spec_verify_rejection(x.logits, x.drafts, None, temperature=1.0, seed=x.seed, offset=50 + i)
        np.testing.assert_array_equal(_np(outs[i][0]), _np(d.out_tokens))
        np.testing.assert_array_equal(_np(outs[i][1]), _np(d.accept_len))
    assert int(_np(st)[0]) == 0


# --------------------------------------------------------------------------------------------
# Trees at small sizes
# --------------------------------------------------------------------------------------------
@pytest.mark.parametrize("V", [5003, 64, 40000])
def test_tree_small(V):
    inp = wl.tree_b48(DEV, B=20, N=8, V=V, seed=V)
    for mode in (0, 1):
        for off in range(3):
            run_tree(inp, mode, offset=off)


def test_tree_wide_and_deep():
    for N, topk, steps in ((16, 15, 8), (32, 4, 31), (64, 8, 14)):
        inp = wl.tree_b48(DEV, B=6, N=N, V=3001, topk=topk, steps=steps, seed=N)
        for mode in (0, 1):
            run_tree(inp, mode)


def test_path_tree_equals_chain_on_gpu():
    inp = wl.chain_b64k7(DEV, B=16, k=6, V=8000, seed=21)
    B, k, V = inp.shape
    tokens = torch.cat([torch.zeros((B, 1), dtype=torch.int32, device=DEV), inp.drafts], 1)
    parents = torch.arange(-1, k, dtype=torch.int32, device=DEV).repeat(B, 1).contiguous()
    c = sv.spec_verify_rejection(inp.logits, inp.drafts, None, temperature=1.0, seed=3, offset=2)
    t = sv.spec_verify_tree(inp.logits, tokens.contiguous(), parents, mode=1, temperature=1.0,
                            seed=3, offset=2)
    assert torch.equal(c.accept_len, t.accept_len)
    assert torch.equal(c.out_tokens, t.out_tokens)


# --------------------------------------------------------------------------------------------
# Faults found in the data: status word, -1 outputs, other requests unaffected
# --------------------------------------------------------------------------------------------
def test_device_status_codes():
    inp = wl.chain_b64k7(DEV, B=6, k=3, V=2000, seed=30)
    d = inp.drafts.clone()
    d[1, 2] = 2000  # out of range
    inp.drafts = d
    r, ref = run_chain(inp, "onehot")
    assert int(_np(r.dev_status)[0]) == 1 and _np(r.accept_len)[1] == -1
    lg = inp.logits.clone()
    lg[3, 1, 17] = float("nan")
    inp2 = wl.ChainInputs("nan", lg, inp.drafts, None, 1.0, 3)
    r, ref = run_chain(inp2, "onehot")
    assert int(_np(r.dev_status)[0]) == 2
    r, ref = run_chain(inp2, "greedy")
    assert int(_np(r.dev_status)[0]) == 2
    lg = inp.logits.clone()
    lg[4, 0, :] = float("-inf")
    inp3 = wl.ChainInputs("neginf", lg, inp.drafts, None, 1.0, 3)
    r, ref = run_chain(inp3, "onehot")
    assert _np(r.accept_len)[4] == -1


def test_tree_status_codes():
    inp = wl.tree_b48(DEV, B=5, N=6, V=1000, seed=2)
    pa = inp.parents.clone()
    pa[1, 3] = 4  # forward parent
    tk = inp.node_tokens.clone()
    tk[2, 1] = 5
    tk[2, 2] = 5
    pa[2, 1] = 0
    pa[2, 2] = 0  # duplicate siblings
    bad = wl.TreeInputs("bad", inp.logits, tk.contiguous(), pa.contiguous(), 1.0, 4)
    r, ref = run_tree(bad, 1)
    assert int(_np(r.dev_status)[0]) == 4
    assert _np(r.accept_len)[1] == -1 and _np(r.accept_len)[2] == -1
    r, ref = run_tree(bad, 0)
    assert int(_np(r.dev_status)[0]) == 3  # duplicates are fine when greedy


# --------------------------------------------------------------------------------------------
# Determinism and workspace reuse
# --------------------------------------------------------------------------------------------
def test_replay_and_workspace_reuse():
    a = wl.chain_b64k7(DEV, B=9, k=5, V=20000, seed=40)
    b = wl.chain_sweep(DEV, B=4, k=2, V=7000, alpha=0.5)
    r1 = sv.spec_verify_rejection(a.logits, a.drafts, None, temperature=1.0, seed=1, offset=9)
    t1, l1 = r1.out_tokens.clone(), r1.accept_len.clone()
    sv.spec_verify_rejection(b.logits, b.drafts, b.q, temperature=1.0, seed=2, offset=0)
    sv.spec_verify_greedy(b.logits, b.drafts)
    r2 = sv.spec_verify_rejection(a.logits, a.drafts, None, temperature=1.0, seed=1, offset=9)
    assert torch.equal(t1, r2.out_tokens) and torch.equal(l1, r2.accept_len)


# --------------------------------------------------------------------------------------------
# The emitted distribution itself (the page's six-token toy, many independent requests)
# --------------------------------------------------------------------------------------------
def test_toy_distribution_on_gpu():
    from scipy import stats

    P = np.array([0.40, 0.25, 0.15, 0.10, 0.07, 0.03])
    Q = np.array([0.20, 0.35, 0.05, 0.25, 0.10, 0.05])
    B, V, calls = 50000, 6, 4
    rng = np.random.default_rng(20261031)
    lt = torch.from_numpy(np.log(np.stack([P, P]))[None].repeat(B, 0).astype(np.float32)).to(DEV)
    qt = torch.from_numpy(np.broadcast_to(Q.astype(np.float32), (B, 1, V)).copy()).to(DEV)
    first, acc = [], []
    for c in range(calls):
        dt = torch.from_numpy(rng.choice(V, size=(B, 1), p=Q).astype(np.int32)).to(DEV)
        r = sv.spec_verify_rejection(lt, dt, qt, temperature=1.0, seed=7, offset=c)
        first.append(_np(r.out_tokens)[:, 0])
        acc.append(_np(r.accept_len) == 1)
    first, acc = np.concatenate(first), np.concatenate(acc)
    n = first.size
    assert abs(acc.mean() - 0.70) < 4 * np.sqrt(0.21 / n)
    assert stats.chisquare(np.bincount(first, minlength=V), P * n).pvalue > 1e-4


def test_rows_with_negative_infinity():
    # -inf logits (masked tokens) are valid as long as a finite logit remains in the row.
    inp = wl.chain_b64k7(DEV, B=6, k=3, V=3000, seed=60)
    lg = inp.logits.clone()
    lg[0, 0, :2000] = float("-inf")
    lg[1, :, ::2] = float("-inf")
    lg[2, 1, 8:] = float("-inf")
    lg[3, 2, :] = float("-inf")
    lg[3, 2, 2999] = 0.0
    inp = wl.ChainInputs("masked", lg, inp.drafts, None, 1.0, 5)
    for mode in ("greedy", "onehot"):
        r, ref = run_chain(inp, mode)
        assert int(_np(r.dev_status)[0]) == 0


def test_one_workspace_across_shapes():
    # A caller-owned workspace, zeroed once, shared by calls of different modes and shapes.
    ws = torch.zeros(sv.spec_verify_workspace_bytes(sv.MODE_REJECTION, 600, 7, 20000),
                     dtype=torch.uint8, device=DEV)
    small = wl.chain_b64k7(DEV, B=3, k=2, V=20000, seed=50)
    big = wl.chain_b64k7(DEV, B=600, k=7, V=517, seed=51)
    tree = wl.tree_b48(DEV, B=7, N=8, V=9000, seed=52)
    for inp in (small, big, small, big):
        r = sv.spec_verify_rejection(inp.logits, inp.drafts, None, temperature=1.0, seed=1,
                                     offset=0, workspace=ws)
        ref = oracle.verify_rejection(wl.to_numpy_logits(inp.logits), _np(inp.drafts), None, 1.0,
                                      1, 0)
        _compare(r.out_tokens, r.accept_len, ref, np.arange(inp.shape[0], dtype=np.int32))
        t = sv.spec_verify_tree(tree.logits, tree.node_tokens, tree.parents, mode=1, seed=2,
                                workspace=ws)
        tref = oracle.verify_tree(wl.to_numpy_logits(tree.logits), _np(tree.node_tokens),
                                  _np(tree.parents), 1, 1.0, 2, 0)
        _compare(t.out_tokens, t.accept_len, tref, np.arange(7, dtype=np.int32))
