"""Pins of the OMP key-selection oracle ("Fast KV Compaction via Attention
Matching", section 2 "Pipeline algorithmique", key selection by orthogonal
matching pursuit) against facts that do not come from the oracle: a pursuit
worked by hand, the closed-form order when the columns have disjoint
supports, forced positions, the least-squares residual property, and the
continuation fits."""
import os

import numpy as np
import pytest

import oracle
from oracle.omp import compact_head_omp, omp_residual, omp_select

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _hand():
    P, orders, resid = [], {}, None
    with open(os.path.join(GOLDEN, "omp_hand_3x3.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            tag, *vals = line.split()
            if tag == "P":
                P.append([float(v) for v in vals])
            elif tag.startswith("order"):
                orders[int(tag[5:])] = [int(v) for v in vals]
            elif tag == "resid2":
                resid = np.array([float(v) for v in vals])
    return np.array(P), orders, resid


def test_hand_worked_pursuit():
    P, orders, resid = _hand()
    for t, want in orders.items():
        order, idx = omp_select(P, t)
        assert order.tolist() == want
        assert idx.tolist() == sorted(want)
    np.testing.assert_allclose(omp_residual(P, orders[2]), resid, atol=1e-12)


def test_disjoint_supports_follow_the_initial_correlations():
    """With columns on disjoint query sets the residual after any set S is 1
    on the rows no chosen column covers, so every later correlation equals the
    initial one: the pursuit takes keys in descending colsum / norm order.
    The column sums and norms are chosen so that this order differs from the
    order by column sum alone."""
    rng = np.random.default_rng(3)
    n_per, T = 5, 7
    P = np.zeros((n_per * T, T))
    for j in range(T):
        col = rng.uniform(0.05, 1.0, n_per)
        col[0] *= 1 + 3 * j                      # spiky columns: large norm for their sum
        P[j * n_per:(j + 1) * n_per, j] = col
    sums, norms = P.sum(axis=0), np.sqrt((P * P).sum(axis=0))
    want = np.argsort(-(sums / norms), kind="stable")
    assert not np.array_equal(want, np.argsort(-sums, kind="stable"))
    order, _ = omp_select(P, T)
    assert order.tolist() == want.tolist()


def test_forced_positions_come_first_and_full_budget_takes_all():
    rng = np.random.default_rng(4)
    P = rng.uniform(0.0, 1.0, (20, 12))
    forced = np.zeros(12, dtype=bool)
    forced[[0, 11]] = True
    order, idx = omp_select(P, 5, forced)
    assert order[:2].tolist() == [0, 11] and len(set(order.tolist())) == 5
    order, idx = omp_select(P, 12)
    assert sorted(order.tolist()) == list(range(12))


def test_residual_is_orthogonal_to_chosen_columns_and_shrinks():
    """Least squares leaves a residual orthogonal to the span of the chosen
    columns, so its norm cannot grow as keys are added."""
    rng = np.random.default_rng(5)
    P = rng.uniform(0.0, 1.0, (30, 16)) ** 3
    order, _ = omp_select(P, 10)
    prev = np.inf
    for s in range(1, 11):
        r = omp_residual(P, order[:s])
        assert np.abs(P[:, order[:s]].T @ r).max() <= 1e-10
        nr = np.linalg.norm(r)
        assert nr <= prev + 1e-12
        prev = nr


def test_never_picks_a_zero_column_while_others_remain():
    P = np.array([[1.0, 0.0, 0.2], [0.5, 0.0, 0.1], [0.0, 0.0, 0.9]])
    order, _ = omp_select(P, 3)
    assert 1 not in order[:2].tolist() and order[-1] == 1


def test_compact_head_omp_fits_its_own_selection():
    """The fits after the pursuit are those of the highest-attention pipeline
    continued from the pursuit's keys: mass matrix = P restricted to the
    chosen columns."""
    rng = np.random.default_rng(6)
    n, T, d, t = 48, 64, 16, 9
    Q, K, V = rng.standard_normal((n, d)), rng.standard_normal((T, d)), rng.standard_normal((T, d))
    r = compact_head_omp(Q, K, V, t)
    scale = 1.0 / np.sqrt(d)
    lse, O, _ = oracle.attention_reference(Q, K, V, scale)
    P = np.exp(Q @ K.T * scale - lse[:, None])
    np.testing.assert_allclose(oracle.mass_matrix(Q, K[r.idx], lse, scale), P[:, r.idx], rtol=1e-12)
    w, beta, _, _, _ = oracle.fit_beta(P[:, r.idx])
    np.testing.assert_allclose(r.w, w, rtol=1e-10, atol=1e-14)
    assert r.order[0] == int(np.argmax(P.sum(axis=0) / np.sqrt((P * P).sum(axis=0))))


def test_rejects_bad_budgets():
    P = np.ones((3, 4))
    with pytest.raises(ValueError):
        omp_select(P, 0)
    with pytest.raises(ValueError):
        omp_select(P, 5)
