"""Pins of the oracle's top-k / top-p filter on p (the target distribution after temperature,
top-k and top-p): the off settings leave softmax unchanged; top-k and top-p keep what their
definitions keep, checked by brute force over prefixes of the sorted vocabulary; ties at a
boundary are kept whole; and a verification with filtered p emits the filtered distribution.

Planting each of these mistakes in a copy of the oracle's filter fails at least one pin: the
(k+1)-th largest logit for the k-th, the top-p mass taken over the whole row instead of the top-k
set, one level kept past the crossing, the level before the crossing as the last one kept, the
boundary level dropped, p not renormalised.  A strict crossing (cum > target for cum >= target)
is not caught: it differs only where a level's running mass equals the target exactly, and the
oracle flags every request within 1e-6 of that as a boundary case."""
import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import chi2


def _row(rng, V, ties=False):
    x = rng.normal(0, 2.0, V)
    if ties:
        x = np.round(x)  # many equal logits
    return x.reshape(1, V)


def test_off_settings_are_plain_softmax(oracle):
    rng = np.random.default_rng(0)
    lg = _row(rng, 50)
    for k, p in ((0, 1.0), (50, 1.0), (-3, 1.0), (77, 1.5)):
        got, _ = oracle.filter_row(lg, 0, 0.8, k, p)
        np.testing.assert_allclose(got, softmax(lg[0] / 0.8), rtol=1e-12)


def test_top_k_brute_force(oracle):
    rng = np.random.default_rng(1)
    for _ in range(30):
        V = int(rng.integers(2, 40))
        lg = _row(rng, V)
        k = int(rng.integers(1, V))
        T = float(rng.uniform(0.3, 2.0))
        got, _ = oracle.filter_row(lg, 0, T, k, 1.0)
        keep = np.argsort(-lg[0], kind="stable")[:k]  # distinct values: exactly the k largest
        want = np.zeros(V)
        want[keep] = softmax(lg[0][keep] / T)
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-300)


def test_top_p_brute_force(oracle):
    """The kept set is the shortest prefix of the descending order whose mass reaches top_p."""
    rng = np.random.default_rng(2)
    for _ in range(40):
        V = int(rng.integers(2, 30))
        lg = _row(rng, V)
        T = float(rng.uniform(0.3, 2.0))
        top_p = float(rng.uniform(0.05, 0.99))
        got, bnd = oracle.filter_row(lg, 0, T, 0, top_p)
        p = softmax(lg[0] / T)
        order = np.argsort(-lg[0], kind="stable")
        for m in range(1, V + 1):
            if p[order[:m]].sum() >= top_p:
                break
        if bnd:
            continue
        want = np.zeros(V)
        want[order[:m]] = p[order[:m]] / p[order[:m]].sum()
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-300)


def test_top_k_then_top_p(oracle):
    rng = np.random.default_rng(3)
    for _ in range(20):
        V = 25
        lg = _row(rng, V)
        k, top_p = int(rng.integers(2, V)), float(rng.uniform(0.2, 0.95))
        got, bnd = oracle.filter_row(lg, 0, 1.0, k, top_p)
        order = np.argsort(-lg[0], kind="stable")[:k]
        pk = softmax(lg[0][order])  # renormalised over the top-k set
        m = int(np.searchsorted(np.cumsum(pk), top_p) + 1)
        if bnd:
            continue
        want = np.zeros(V)
        want[order[:m]] = pk[:m] / pk[:m].sum()
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-300)


def test_ties_at_the_boundary_are_kept_whole(oracle):
    lg = np.array([[3.0, 1.0, 3.0, 2.0, 1.0, 0.0]])
    got, _ = oracle.filter_row(lg, 0, 1.0, 1, 1.0)  # the largest value is shared by 0 and 2
    np.testing.assert_allclose(got, [0.5, 0, 0.5, 0, 0, 0])
    got, _ = oracle.filter_row(lg, 0, 1.0, 4, 1.0)  # 4th largest is 1.0: tokens 1 and 4 both kept
    assert (got > 0).sum() == 5 and got[5] == 0.0
    got, _ = oracle.filter_row(lg, 0, 1.0, 0, 0.3)  # the top level alone holds 2 e^3 / Z > 0.3
    assert (got > 0).tolist() == [True, False, True, False, False, False]


def test_verification_emits_the_filtered_distribution(oracle):
    """Many requests with the same row and one-hot drafts: the first emitted token's frequencies
    follow the filtered p (chi-square), whatever the draft."""
    rng = np.random.default_rng(4)
    V, B = 12, 6000
    row = rng.normal(0, 1.5, V)
    lg = np.broadcast_to(row, (B, 2, V)).copy()
    drafts = rng.integers(0, V, (B, 1)).astype(np.int32)
    tk, tp = np.full(B, 6, np.int32), np.full(B, 0.8)
    r = oracle.verify_ex(lg, drafts, None, np.ones(B), seed=7, offset=0, top_k=tk, top_p=tp)
    want, _ = oracle.filter_row(lg[0], 0, 1.0, 6, 0.8)
    counts = np.bincount(r["out_tokens"][:, 0], minlength=V)
    assert counts[want == 0].sum() == 0
    e = want[want > 0] * B
    stat = ((counts[want > 0] - e) ** 2 / e).sum()
    assert stat < chi2.ppf(0.999, (want > 0).sum() - 1)


def test_invalid_top_p(oracle):
    lg = np.zeros((2, 3, 5))
    with pytest.raises(RuntimeError):
        oracle.verify_ex(lg, np.zeros((2, 2), np.int32), None, [1.0, 1.0], 0, 0, top_p=[0.5, 0.0])
