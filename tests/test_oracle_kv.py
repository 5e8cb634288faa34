"""Pins of the oracle's KV compaction after tree verification (the accepted path's KV rows moved
to contiguous positions after the committed prefix; the committed length advanced by the
accepted nodes plus one)."""
import numpy as np


def _random_tree(rng, N):
    parents = np.full(N, -1, np.int32)
    for j in range(1, N):
        parents[j] = rng.integers(0, j)
    return parents


def _random_path(rng, parents):
    N = len(parents)
    path, cur = [0], 0
    while True:
        ch = [j for j in range(1, N) if parents[j] == cur]
        if not ch or rng.random() < 0.3:
            return path
        cur = int(rng.choice(ch))
        path.append(cur)


def _case(rng, B=6, N=8, max_pos=64, row=5):
    num_slots = B * max_pos
    perm = rng.permutation(num_slots).astype(np.int32)
    slot_table = perm.reshape(B, max_pos)
    committed = rng.integers(0, max_pos - N, B).astype(np.int32)
    accept_index = np.full((B, N), -1, np.int32)
    accept_len = np.zeros(B, np.int32)
    for b in range(B):
        path = _random_path(rng, _random_tree(rng, N))
        accept_index[b, : len(path)] = path
        accept_len[b] = len(path) - 1
    pool = rng.normal(size=(num_slots, row)).astype(np.float32)
    return pool, slot_table, committed, accept_index, accept_len


def test_the_committed_sequence_reads_the_accepted_path(oracle):
    rng = np.random.default_rng(0)
    for _ in range(20):
        pool, st, c, ai, al = _case(rng)
        before = pool.copy()
        new, status = oracle.kv_compact(pool, st, c, ai, al)
        assert not status.any()
        for b in range(len(c)):
            # Brute force: what attention reads at positions c .. c + L is the path's rows.
            for i in range(al[b] + 1):
                np.testing.assert_array_equal(pool[st[b, c[b] + i]], before[st[b, c[b] + ai[b, i]]])
            assert new[b] == c[b] + al[b] + 1
        # Rows of the committed prefix and of other requests' positions below theirs are untouched.
        for b in range(len(c)):
            for pos in range(c[b]):
                np.testing.assert_array_equal(pool[st[b, pos]], before[st[b, pos]])


def test_a_chain_moves_nothing(oracle):
    rng = np.random.default_rng(1)
    pool, st, c, ai, al = _case(rng)
    N = ai.shape[1]
    for b in range(len(c)):
        al[b] = rng.integers(0, N)
        ai[b] = -1
        ai[b, : al[b] + 1] = np.arange(al[b] + 1)
    before = pool.copy()
    new, status = oracle.kv_compact(pool, st, c, ai, al)
    np.testing.assert_array_equal(pool, before)
    np.testing.assert_array_equal(new, c + al + 1)


def test_faulted_and_out_of_range_requests_are_left_alone(oracle):
    rng = np.random.default_rng(2)
    pool, st, c, ai, al = _case(rng)
    al[0] = -1
    c[1] = st.shape[1] - 2  # the tree would run past the slot table
    st[2, c[2] + ai[2, al[2]]] = pool.shape[0] + 5  # a slot outside the pool
    before = pool.copy()
    new, status = oracle.kv_compact(pool, st, c, ai, al)
    assert list(status[:3]) == [0, oracle.KV_BAD_POSITION, oracle.KV_BAD_SLOT]
    assert new[0] == c[0] and new[1] == c[1] and new[2] == c[2]
    for b in range(3):
        for pos in range(st.shape[1]):
            s = st[b, pos]
            if 0 <= s < pool.shape[0]:
                np.testing.assert_array_equal(pool[s], before[s])


def test_planes_move_together_and_bad_indices_are_rejected(oracle):
    rng = np.random.default_rng(3)
    pool, st, c, ai, al = _case(rng)
    stack = np.stack([pool, pool * 2.0, -pool])  # three planes (layers' K or V)
    ref = pool.copy()
    new2, _ = oracle.kv_compact(ref, st, c, ai, al)
    new3, status = oracle.kv_compact(stack, st, c, ai, al)
    assert not status.any()
    np.testing.assert_array_equal(new2, new3)
    np.testing.assert_array_equal(stack[0], ref)
    np.testing.assert_array_equal(stack[1], ref * 2.0)
    np.testing.assert_array_equal(stack[2], -ref)
    # An accept_index entry outside [0, N) on the accepted path is a position error.
    b = int(np.argmax(al))
    assert al[b] >= 1
    ai2 = ai.copy()
    ai2[b, al[b]] = ai.shape[1]
    before = pool.copy()
    new, status = oracle.kv_compact(pool, st, c, ai2, al)
    assert status[b] == oracle.KV_BAD_POSITION and new[b] == c[b]
    for pos in range(st.shape[1]):
        np.testing.assert_array_equal(pool[st[b, pos]], before[st[b, pos]])
