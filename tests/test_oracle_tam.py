"""Pins of the thought-aware compaction oracle ("Thought-Aware KV Cache
Compaction" explainer, section 2: adaptive budgets t_i ~ sqrt(w_i) n_i,
pivot tokens kept exactly with zero bias) against facts that do not come
from the oracle: allocations worked by hand, thresholds on hand-made
attention, library solvers (scipy NNLS, numpy least squares) on the
augmented systems of the fixed-pivot fits, and the reduction to Attention
Matching with one segment and no pivots."""
import os

import numpy as np
import pytest
from scipy.optimize import nnls

import oracle
from oracle.tam import (allocate_budgets, compact_head_tam, detect_pivots, fit_beta_fixed, fit_values_fixed,
                        select_segments, window_attention)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _alloc_cases():
    with open(os.path.join(GOLDEN, "tam_allocation.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            w, n, tot, want = (part.split() for part in line.split("|"))
            yield [float(x) for x in w], [int(x) for x in n], int(tot[0]), [int(x) for x in want]


@pytest.mark.parametrize("case", list(_alloc_cases()))
def test_allocation_worked_by_hand(case):
    w, n, tot, want = case
    got = allocate_budgets(w, n, tot)
    assert got.tolist() == want
    assert int(got.sum()) == tot and np.all(got <= np.array(n)) and np.all(got >= 0)


def test_allocation_is_proportional_when_exact():
    # sqrt(w) n = 3*4, 1*8, 2*2 = 12, 8, 4 -> 24 units split 12 : 8 : 4
    got = allocate_budgets([9, 1, 4], [40, 80, 20], 24)
    assert got.tolist() == [12, 8, 4]


def test_pivot_threshold_by_hand():
    alpha = np.array([0.1, 0.5, 0.1, 0.3])          # mean 0.25
    assert detect_pivots(alpha, 1.5).tolist() == [False, True, False, False]
    assert detect_pivots(alpha, 1.0).tolist() == [False, True, False, True]


def test_window_attention_is_a_mean_of_distributions():
    rng = np.random.default_rng(1)
    K = rng.standard_normal((30, 8))
    a = window_attention(np.zeros((5, 8)), K, 0.3)
    np.testing.assert_allclose(a, np.full(30, 1 / 30), rtol=1e-14)      # q = 0: uniform
    a = window_attention(rng.standard_normal((7, 8)), K, 0.3)
    assert abs(a.sum() - 1.0) < 1e-12 and np.all(a > 0)


def test_segment_selection_by_hand():
    score = np.array([0.2, 0.9, 0.5, 0.1, 0.0, 0.3])
    piv = np.array([False, False, False, False, True, False])
    idx = select_segments(score, [0, 3, 6], [1, 2], piv)
    # segment 0 keeps its best key (1); segment 1 keeps pivot 4 and keys 5, 3
    assert idx.tolist() == [1, 3, 4, 5]


def _tiny(seed, n=40, t=9):
    rng = np.random.default_rng(seed)
    Ap = rng.uniform(0.0, 0.2, (n, t)) ** 2
    piv = np.zeros(t, dtype=bool)
    piv[[1, 6]] = True
    return Ap, piv


def test_fixed_pivot_nnls_matches_scipy_on_the_augmented_system():
    Ap, piv = _tiny(2)
    w, beta, mu = fit_beta_fixed(Ap, piv)
    assert np.all(w[piv] == 1.0) and np.all(beta[piv] == 0.0)
    A = Ap[:, ~piv]
    tgt = 1.0 - Ap[:, piv].sum(axis=1)
    aug = np.vstack([A, np.sqrt(mu) * np.eye(A.shape[1])])
    rhs = np.concatenate([tgt, np.sqrt(mu) * np.ones(A.shape[1])])
    ref, _ = nnls(aug, rhs)
    np.testing.assert_allclose(w[~piv], ref, rtol=1e-7, atol=1e-9)
    assert mu == pytest.approx(1e-2 * np.trace(Ap.T @ Ap) / Ap.shape[1], rel=1e-14)


def test_fixed_pivot_nnls_without_pivots_is_the_plain_fit():
    Ap, _ = _tiny(3)
    w, _, _ = fit_beta_fixed(Ap, np.zeros(Ap.shape[1], dtype=bool))
    w0, *_ = oracle.fit_beta(Ap)
    np.testing.assert_allclose(w, w0, rtol=1e-12, atol=1e-15)


def test_fixed_pivot_values_match_lstsq_on_the_augmented_system():
    rng = np.random.default_rng(4)
    Ap, piv = _tiny(4)
    w = rng.uniform(0.5, 2.0, Ap.shape[1])
    X = oracle.biased_softmax(Ap, w)
    O = rng.standard_normal((Ap.shape[0], 5))
    Vs = rng.standard_normal((Ap.shape[1], 5))
    Cv, lam = fit_values_fixed(X, O, Vs, piv)
    np.testing.assert_array_equal(Cv[piv], Vs[piv])
    A = X[:, ~piv]
    aug = np.vstack([A, np.sqrt(lam) * np.eye(A.shape[1])])
    rhs = np.vstack([O - X[:, piv] @ Vs[piv], np.sqrt(lam) * Vs[~piv]])
    ref, *_ = np.linalg.lstsq(aug, rhs, rcond=None)
    np.testing.assert_allclose(Cv[~piv], ref, rtol=1e-9, atol=1e-11)


def test_one_segment_without_pivots_is_attention_matching():
    rng = np.random.default_rng(5)
    n, T, d, t = 48, 96, 16, 12
    Q, K, V = rng.standard_normal((n, d)), rng.standard_normal((T, d)), rng.standard_normal((T, d))
    Qw = rng.standard_normal((6, d))
    r = compact_head_tam(Q, K, V, Qw, [0, T], t, c=1e9)
    r0 = oracle.compact_head(Q, K, V, t)
    assert not r.pivots.any() and r.seg_budgets.tolist() == [t]
    assert r.idx.tolist() == r0.idx.tolist()
    np.testing.assert_allclose(r.w, r0.w, rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(r.Cv, r0.Cv, rtol=1e-10, atol=1e-12)


def test_pivots_are_kept_with_zero_bias_and_their_values():
    rng = np.random.default_rng(6)
    n, T, d = 48, 120, 16
    Q, K, V = rng.standard_normal((n, d)), rng.standard_normal((T, d)), rng.standard_normal((T, d))
    K[[7, 50]] *= 4.0                                   # strong keys: pivots for a query near them
    Qw = np.vstack([K[7], K[50], rng.standard_normal((4, d))])
    r = compact_head_tam(Q, K, V, Qw, [0, 40, 80, 120], 20, c=5.0)
    assert r.pivots.sum() >= 1
    kept_p = r.pivots[r.idx]
    assert np.all(r.beta[kept_p] == 0.0)
    np.testing.assert_array_equal(r.Cv[kept_p], V[r.idx[kept_p]])
    assert set(np.flatnonzero(r.pivots)) <= set(r.idx.tolist())
    assert len(r.idx) == 20 and int(r.seg_budgets.sum()) == 20 - int(r.pivots.sum())
