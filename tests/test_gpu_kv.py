"""Parity of the CUDA KV compaction after tree verification (spec_verify_kv_compact, through its C
ABI) with the oracle: the pool's bytes, the committed lengths and the status must match exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_verify_gb300 as sv
from speculative_decoding_verification_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
DEV_CODE = {oracle.KV_OK: 0, oracle.KV_BAD_POSITION: sv.binding.DEV_BAD_KV_POSITION,
            oracle.KV_BAD_SLOT: sv.binding.DEV_BAD_KV_SLOT}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_verify_gb300 import _build

    _build.build()
    torch.cuda.set_device(DEV)


def _np(t):
    return t.detach().cpu().numpy()


def run_kv(inp: wl.KVInputs, stacked=True, pool=None):
    """Compact on the GPU and in the oracle from the same inputs; compare everything."""
    pool = inp.pool if pool is None else pool
    ref_pool = _np(pool).copy()
    new_ref, status = oracle.kv_compact(ref_pool, _np(inp.slot_table), _np(inp.committed),
                                        _np(inp.accept_index), _np(inp.accept_len))
    c_out, dev_status = sv.spec_verify_kv_compact(pool, inp.slot_table, inp.committed,
                                                  inp.accept_index, inp.accept_len, stacked=stacked)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_np(c_out), new_ref)
    assert int(_np(dev_status)[0]) == max(DEV_CODE[int(s)] for s in status)
    got = _np(pool)
    if not np.array_equal(got, ref_pool):
        bad = np.argwhere(got != ref_pool)
        raise AssertionError(f"{len(bad)} pool elements differ, first at {bad[0].tolist()}")
    return new_ref, status


@pytest.mark.parametrize("row_bytes", [16, 48, 2048, 16400])
def test_kv_random_paths_one_plane(row_bytes):
    for seed in range(3):
        inp = wl.kv_paged(DEV, seed=seed, B=9, N=8, planes=1, row_bytes=row_bytes, max_pos=40)
        run_kv(wl.KVInputs(inp.name, inp.pool[0], inp.slot_table, inp.committed,
                           inp.accept_index, inp.accept_len), stacked=False)


@pytest.mark.parametrize("planes,row_bytes", [(5, 272), (64, 2048), (3, 65536)])
def test_kv_stacked_planes(planes, row_bytes):
    inp = wl.kv_paged(DEV, seed=planes, B=6, N=8, planes=planes, row_bytes=row_bytes, max_pos=24)
    new, status = run_kv(inp)
    assert not status.any()
    np.testing.assert_array_equal(new, _np(inp.committed) + _np(inp.accept_len) + 1)


def test_kv_planes_with_gaps():
    """Planes need not be back to back: a view into a larger buffer keeps its plane stride, and
    the bytes between planes stay untouched."""
    inp = wl.kv_paged(DEV, seed=11, B=5, N=8, planes=4, row_bytes=96, max_pos=20)
    P, S, R = inp.pool.shape
    big = torch.randint(-100, 100, (P, S + 7, R), dtype=torch.int16, device=DEV)
    big[:, :S] = inp.pool
    tail = big[:, S:].clone()
    view = big[:, :S]
    assert not view.is_contiguous() and view[0].is_contiguous()
    run_kv(inp, pool=view)
    assert torch.equal(big[:, S:], tail)


def test_kv_long_paths_and_wide_trees():
    for N in (2, 17, 64):
        inp = wl.kv_paged(DEV, seed=100 + N, B=7, N=N, planes=2, row_bytes=144, max_pos=N + 9,
                          topk=N, steps=N, p_stop=0.05)
        run_kv(inp)
    # N = 1: the root alone, nothing moves, committed grows by one.
    inp = wl.kv_paged(DEV, seed=5, B=4, N=1, planes=2, row_bytes=32, max_pos=3)
    new, _ = run_kv(inp)
    np.testing.assert_array_equal(new, _np(inp.committed) + 1)


def test_kv_indices_off_a_path_keep_the_sequential_order():
    """accept_index entries that do not form a root-to-node path (repeats, going back up) make a
    step read a row an earlier step wrote; the result must still be that of copying the steps
    one by one in order, as the oracle does."""
    inp = wl.kv_paged(DEV, seed=41, B=12, N=8, planes=3, row_bytes=80, max_pos=20)
    rng = np.random.default_rng(41)
    ai = _np(inp.accept_index).copy()
    al = _np(inp.accept_len).copy()
    for b in range(12):
        al[b] = rng.integers(1, 8)
        ai[b, : al[b] + 1] = rng.integers(0, 8, al[b] + 1)
    ai[0, :4] = [0, 2, 1, 3]  # step 2 reads position 1, which step 1 wrote
    al[0] = 3
    t = lambda a: torch.from_numpy(a).to(DEV)  # noqa: E731
    run_kv(wl.KVInputs("off_path", inp.pool, inp.slot_table, inp.committed, t(ai), t(al)))


def test_kv_status_codes_leave_requests_alone():
    inp = wl.kv_paged(DEV, seed=21, B=8, N=8, planes=3, row_bytes=64, max_pos=30, extra_slots=4)
    al, c = inp.accept_len.clone(), inp.committed.clone()
    ai, st = inp.accept_index.clone(), inp.slot_table.clone()
    S = int(inp.pool.shape[1])
    al[0] = -1                                      # a request the verifier faulted
    c[1] = 30 - 7                                   # the tree would run past the slot table
    st[2, int(c[2]) + int(ai[2, int(al[2])])] = S + 3  # a path slot outside the pool
    st[3, int(c[3])] = -2                           # the root's destination slot is negative
    ai[4, int(al[4])] = 8                           # a path entry outside [0, N)
    ai[5, int(al[5])] = 8                           # both errors: the position error is reported
    st[5, int(c[5])] = S
    al[6] = 8                                       # accept_len >= N
    bad = wl.KVInputs("bad", inp.pool, st, c, ai, al)
    new, status = run_kv(bad)
    P_, S_ = oracle.KV_BAD_POSITION, oracle.KV_BAD_SLOT
    assert list(status) == [0, P_, S_, S_, P_, P_, P_, 0]
    np.testing.assert_array_equal(new[:7], _np(c)[:7])
    # Only position errors: the slot code is not reached.
    ok = wl.kv_paged(DEV, seed=22, B=4, N=8, planes=1, row_bytes=32, max_pos=12)
    c2 = ok.committed.clone()
    c2[2] = -1
    new, status = run_kv(wl.KVInputs("pos", ok.pool, ok.slot_table, c2, ok.accept_index,
                                     ok.accept_len))
    assert list(status) == [0, 0, oracle.KV_BAD_POSITION, 0]


def test_kv_after_tree_verification():
    """The whole bookkeeping step: each side compacts with the accepted path its own tree
    verifier found (GPU: spec_verify_tree; oracle: verify_tree); requests the oracle flags as
    boundary draws are left out of the comparison."""
    tree = wl.tree_b48(DEV, V=5003)
    B, N, V = tree.shape
    kv = wl.kv_paged(DEV, seed=31, B=B, N=N, planes=4, row_bytes=256, max_pos=48)
    lg = wl.to_numpy_logits(tree.logits)
    for mode in (0, 1):
        r = sv.spec_verify_tree(tree.logits, tree.node_tokens, tree.parents, mode=mode,
                                temperature=tree.temperature, seed=tree.seed)
        ref = oracle.verify_tree(lg, _np(tree.node_tokens), _np(tree.parents), mode,
                                 tree.temperature, tree.seed, 0)
        pool = kv.pool.clone()
        host = _np(pool).copy()
        new_ref, st_ref = oracle.kv_compact(host, _np(kv.slot_table), _np(kv.committed),
                                            ref["accept_index"], ref["accept_len"])
        c_out, dev_status = sv.spec_verify_kv_compact(pool, kv.slot_table, kv.committed,
                                                      r.accept_index, r.accept_len, stacked=True)
        torch.cuda.synchronize()
        assert not st_ref.any() and int(_np(dev_status)[0]) == 0
        ok = ~ref["boundary"].astype(bool)
        assert (~ok).sum() <= 1
        np.testing.assert_array_equal(_np(c_out)[ok], new_ref[ok])
        got = _np(pool)
        st = _np(kv.slot_table)
        for b in np.flatnonzero(ok):
            np.testing.assert_array_equal(got[:, st[b]], host[:, st[b]])
        if mode == 0:
            assert len(set(ref["accept_len"].tolist())) >= 3


def test_kv_full_size_sampled():
    """Llama-3-8B-sized cache (64 planes of 2048-byte rows), B=48, N=8, 512 positions each: the
    rows of a sample of requests, plus every committed length, against the oracle run on just
    those requests' slots."""
    inp = wl.kv_paged(DEV)
    before = {}
    st = _np(inp.slot_table)
    sample = [0, 7, 23, 47]
    for b in sample:
        before[b] = _np(inp.pool[:, torch.from_numpy(st[b]).long().to(DEV)]).copy()
    c_out, dev_status = sv.spec_verify_kv_compact(inp.pool, inp.slot_table, inp.committed,
                                                  inp.accept_index, inp.accept_len, stacked=True)
    torch.cuda.synchronize()
    assert int(_np(dev_status)[0]) == 0
    np.testing.assert_array_equal(_np(c_out), _np(inp.committed) + _np(inp.accept_len) + 1)
    for b in sample:
        # The oracle on request b alone, with its own positions mapped to slots 0..max_pos-1.
        local = before[b].copy()
        new, status = oracle.kv_compact(local, np.arange(st.shape[1], dtype=np.int32)[None],
                                        _np(inp.committed)[b:b + 1], _np(inp.accept_index)[b:b + 1],
                                        _np(inp.accept_len)[b:b + 1])
        got = _np(inp.pool[:, torch.from_numpy(st[b]).long().to(DEV)])
        np.testing.assert_array_equal(got, local)
