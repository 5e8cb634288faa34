"""Pins of the oracle's counter-based RNG (Philox4x32-10, Salmon et al. SC'11)."""
import json
import os

import numpy as np
import pytest
from scipy import stats


def test_known_answer_vectors(oracle, golden_dir):
    kat = json.load(open(os.path.join(golden_dir, "philox4x32_10_kat.json")))
    for vec in kat["vectors"]:
        ctr = [int(w, 16) for w in vec["ctr"]]
        key = [int(w, 16) for w in vec["key"]]
        out = [int(w, 16) for w in vec["out"]]
        assert list(oracle.philox4x32_10(ctr, key)) == out


def test_u01_is_top_24_bits(oracle):
    assert oracle.u01(0) == 0.0
    assert oracle.u01(0xFF) == 0.0
    assert oracle.u01(0x100) == 2.0 ** -24
    assert oracle.u01(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle.u01(0x80000000) == 0.5


def test_uniform_pair_uses_words_0_and_1(oracle):
    seed, offset, slot, req = 0x1234_5678_9ABC_DEF0, 0x0000_0007_0000_0003, 5, 17
    words = oracle.philox4x32_10([slot, req, offset & 0xFFFFFFFF, offset >> 32],
                                 [seed & 0xFFFFFFFF, seed >> 32])
    u, v = oracle.uniform_pair(seed, offset, slot, req)
    assert u == (int(words[0]) >> 8) * 2.0 ** -24
    assert v == (int(words[1]) >> 8) * 2.0 ** -24


@pytest.mark.parametrize("seed", [20261031, 7])
def test_uniformity_and_pair_independence(oracle, seed):
    n_slot, n_req = 50, 2000
    us = np.empty(n_slot * n_req)
    vs = np.empty(n_slot * n_req)
    i = 0
    for s in range(n_slot):
        for b in range(n_req):
            us[i], vs[i] = oracle.uniform_pair(seed, 3, s, b)
            i += 1
    for x in (us, vs):
        counts = np.histogram(x, bins=50, range=(0, 1))[0]
        assert stats.chisquare(counts).pvalue > 1e-4
    joint = np.histogram2d(us, vs, bins=10, range=[[0, 1], [0, 1]])[0].ravel()
    assert stats.chisquare(joint).pvalue > 1e-4
    # Different offsets give unrelated streams.
    u2 = np.array([oracle.uniform_pair(seed, 4, 0, b)[0] for b in range(n_req)])
    assert abs(np.corrcoef(us[:n_req], u2)[0, 1]) < 0.1
