"""The range-checked build (-DSV_DEBUG): every global-memory access of every kernel is checked
against the extent of the array it falls in, and a violation is recorded rather than followed
(no trap, no assert).  Small cases of every entry point run through the debug build must record
no violation and give outputs bit-identical to the release build's (which the parity tests
compare with the oracle).  This stands in for a memory checker."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_verify_gb300 as sv
from speculative_decoding_verification_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def debug_lib():
    torch.cuda.set_device(DEV)
    sv.load_library()
    return sv.load_debug_library()


def _cases():
    """(name, callable returning a tuple of output tensors) for small cases of every entry point;
    the callables use the module's wrappers, so they run on whichever build is routed in."""
    out = []
    tiny = wl.chain_tiny(DEV)
    out.append(("standard tiny", lambda: sv.spec_verify_rejection(tiny.logits, tiny.drafts, tiny.q, temperature=1.0,
                                                                   seed=tiny.seed, offset=1, want_probs=True)))
    out.append(("greedy tiny", lambda: sv.spec_verify_greedy(tiny.logits, tiny.drafts)))
    for V in (4099, 131):
        c = wl.chain_b64k7(DEV, B=6, k=7, V=V, seed=V)
        out.append((f"one-hot V={V}", lambda c=c: sv.spec_verify_rejection(c.logits, c.drafts, None, temperature=0.8,
                                                                          seed=3, offset=2, want_probs=True)))
        out.append((f"greedy V={V}", lambda c=c: sv.spec_verify_greedy(c.logits, c.drafts)))
        out.append((f"block one-hot V={V}", lambda c=c: sv.spec_verify_block(c.logits, c.drafts, None, temperature=1.0,
                                                                            seed=3, offset=2)))
    q = wl.chain_sweep(DEV, B=5, k=4, V=3001, alpha=0.5)
    out.append(("standard with q", lambda: sv.spec_verify_rejection(q.logits, q.drafts, q.q, temperature=1.0, seed=4,
                                                                    offset=0, want_probs=True)))
    out.append(("block with q", lambda: sv.spec_verify_block(q.logits, q.drafts, q.q, temperature=1.0, seed=4,
                                                             offset=0)))
    # An unaligned logits base (every row's head and tail read element by element).
    base = wl.chain_b64k7(DEV, B=3, k=3, V=10007, seed=5)
    buf = torch.empty(3 * 4 * 10007 + 8, dtype=torch.bfloat16, device=DEV)
    view = buf[3:3 + 3 * 4 * 10007].view(3, 4, 10007)
    view.copy_(base.logits)
    out.append(("unaligned", lambda: sv.spec_verify_rejection(view, base.drafts, None, temperature=1.0, seed=1,
                                                              offset=0)))
    tk3 = torch.tensor([1, 60, 512], dtype=torch.int32, device=DEV)
    tp3 = torch.tensor([0.9, 1.0, 0.5], device=DEV)
    out.append(("unaligned top-k top-p", lambda: sv.spec_verify_rejection_ex(view, base.drafts, None, top_k=tk3,
                                                                             top_p=tp3, seed=1, offset=0)))
    tr = wl.tree_b48(DEV, B=5, N=8, V=5003, seed=6)
    for mode in (0, 1):
        out.append((f"tree mode {mode}", lambda mode=mode: sv.spec_verify_tree(
            tr.logits, tr.node_tokens, tr.parents, mode=mode, temperature=1.0, seed=7, offset=0)))
    v = wl.chain_b64k7(DEV, B=6, k=5, V=3001, seed=8)
    temps = torch.tensor([0.0, 1.0, 0.7, 0.0, 1.3, 1.0], device=DEV)
    tk = torch.tensor([1, 5, 0, 40, 3000, 2], dtype=torch.int32, device=DEV)
    tp = torch.tensor([1.0, 0.9, 0.5, 1.0, 0.2, 0.95], device=DEV)
    out.append(("mixed temperatures", lambda: sv.spec_verify_rejection_ex(v.logits, v.drafts, None, temperatures=temps,
                                                                          seed=9, offset=1)))
    out.append(("top-k top-p", lambda: sv.spec_verify_rejection_ex(v.logits, v.drafts, None, top_k=tk, top_p=tp,
                                                                   seed=9, offset=1)))
    out.append(("relaxed thresholds", lambda: sv.spec_verify_rejection_ex(
        v.logits, v.drafts, None, threshold_single=0.5, threshold_acc=0.5, seed=9, offset=1)))
    out.append(("tree top-k", lambda: sv.spec_verify_tree_ex(tr.logits, tr.node_tokens, tr.parents, top_k=tk[:1].repeat(5),
                                                             seed=9)))
    kv = wl.kv_paged(DEV, B=5, N=8, planes=3, row_bytes=96, max_pos=20)

    def kv_call():
        pool = kv.pool.clone()
        c, st = sv.spec_verify_kv_compact(pool, kv.slot_table, kv.committed, kv.accept_index, kv.accept_len,
                                          stacked=True)
        return (pool, c, st)

    out.append(("kv compaction", kv_call))
    conf = torch.rand((40, 7), generator=torch.Generator(device=DEV).manual_seed(3), device=DEV)
    cost = 1e-3 + torch.arange(40 * 7 + 1, device=DEV, dtype=torch.float64) * 1e-5
    out.append(("adaptive budget", lambda: sv.spec_verify_plan_budget(conf, cost)))
    return out


def _tensors(r):
    if isinstance(r, torch.Tensor):
        return [r]
    if isinstance(r, (tuple, list)):
        return [t for x in r for t in _tensors(x)]
    if hasattr(r, "_asdict"):
        return [t for x in r._asdict().values() for t in _tensors(x)]
    return []


def test_debug_build_checks_every_access_and_matches_release(debug_lib):
    cases = _cases()
    release = {}
    for name, fn in cases:
        release[name] = [t.detach().cpu().clone() for t in _tensors(fn())]
    torch.cuda.synchronize()
    assert sv.spec_verify_debug_fault() == 0  # a release build records nothing
    assert sv.spec_verify_debug_fault(debug_lib) == 0
    with sv.using_library(debug_lib):
        for name, fn in cases:
            got = [t.detach().cpu() for t in _tensors(fn())]
            torch.cuda.synchronize()
            fault = sv.spec_verify_debug_fault(debug_lib)
            assert fault == 0, f"{name}: range check {fault >> 48 & 0x7fff} failed at index {fault & (2**48 - 1)}"
            assert len(got) == len(release[name]), name
            for a, b in zip(release[name], got):
                assert torch.equal(a, b), name
