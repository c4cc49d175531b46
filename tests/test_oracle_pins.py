"""Pins of the float64 oracle against facts that do not come from it.

Each test names what it pins: brute force on tiny inputs (pure-Python loops
with math.exp), closed forms, the KKT conditions of NNLS, exhaustive support
enumeration, library solvers on special cases, and the page's q = 0 example
("Fast KV Compaction via Attention Matching", section 2, "Objectif principal").
"""
import itertools
import math
import os

import numpy as np
import pytest
from scipy.optimize import nnls as scipy_nnls

import oracle
from oracle import am

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, *shape, s=1.0):
    return rng.standard_normal(shape) * s


# ------------------------------------------------------------- step 1
def test_attention_matches_pure_python_softmax():
    """lse and O against a per-query loop with math.exp/math.log (brute force)."""
    rng = np.random.default_rng(1)
    n, T, d = 5, 7, 3
    Q, K, V = _rand(rng, n, d, s=2.0), _rand(rng, T, d, s=2.0), _rand(rng, T, 2)
    scale = 1 / math.sqrt(d)
    lse, O, colsq = oracle.attention_reference(Q, K, V, scale, row_chunk=2)
    for q in range(n):
        logits = [sum(Q[q, k] * K[j, k] for k in range(d)) * scale for j in range(T)]
        mass = sum(math.exp(x) for x in logits)
        assert abs(lse[q] - math.log(mass)) < 1e-12
        for c in range(2):
            o = sum(math.exp(logits[j]) / mass * V[j, c] for j in range(T))
            assert abs(O[q, c] - o) < 1e-12
    for j in range(T):
        s2 = 0.0
        for q in range(n):
            logits = [sum(Q[q, k] * K[i, k] for k in range(d)) * scale for i in range(T)]
            p = math.exp(logits[j]) / sum(math.exp(x) for x in logits)
            s2 += p * p
        assert abs(colsq[j] - s2) < 1e-12


def test_attention_closed_form_zero_keys():
    """K = 0: every logit is 0, so lse = log T, O = mean of V, P = 1/T."""
    rng = np.random.default_rng(2)
    n, T, d = 6, 11, 4
    Q, V = _rand(rng, n, d), _rand(rng, T, 3)
    lse, O, colsq = oracle.attention_reference(Q, np.zeros((T, d)), V, 0.5)
    np.testing.assert_allclose(lse, np.log(T), rtol=0, atol=1e-14)
    np.testing.assert_allclose(O, np.tile(V.mean(0), (n, 1)), rtol=0, atol=1e-14)
    np.testing.assert_allclose(oracle.key_scores(colsq, n), 1.0 / T, rtol=1e-14)


def test_attention_huge_logits_stable():
    """Logits of +-1000 (far outside exp's range) still give the exact
    one-hot softmax: the log-sum-exp shift is in place."""
    Q = np.array([[1000.0, 0.0]])
    K = np.array([[1.0, 0.0], [0.999, 0.0], [-1.0, 0.0]])
    V = np.array([[1.0], [2.0], [3.0]])
    lse, O, _ = oracle.attention_reference(Q, K, V, 1.0)
    assert abs(lse[0] - (1000.0 + math.log1p(math.exp(-1.0)))) < 1e-9
    assert abs(O[0, 0] - (1.0 + 2.0 * math.exp(-1.0)) / (1 + math.exp(-1.0))) < 1e-12


# ------------------------------------------------------------- step 2
def test_score_is_rms_of_attention_weights():
    rng = np.random.default_rng(3)
    n, T, d = 4, 6, 2
    Q, K = _rand(rng, n, d), _rand(rng, T, d)
    lse, _, colsq = oracle.attention_reference(Q, K, np.zeros((T, 1)), 0.7)
    score = oracle.key_scores(colsq, n)
    for j in range(T):
        ps = []
        for q in range(n):
            lg = [float(Q[q] @ K[i]) * 0.7 for i in range(T)]
            ps.append(math.exp(lg[j]) / sum(math.exp(x) for x in lg))
        assert abs(score[j] - math.sqrt(sum(p * p for p in ps) / n)) < 1e-14


@pytest.mark.parametrize("seed", range(6))
def test_top_t_brute_force_subsets(seed):
    """Top-t = the t-subset with the largest float32 score sum, ties to the
    lexicographically smallest index set (many ties: integer scores)."""
    rng = np.random.default_rng(seed)
    T = int(rng.integers(5, 12))
    t = int(rng.integers(1, T + 1))
    score = rng.integers(0, 4, size=T).astype(np.float64) / 4.0
    idx = oracle.select_top_t(score, t)
    best = None
    for sub in itertools.combinations(range(T), t):
        s = sum(float(np.float32(score[j])) for j in sub)
        if best is None or s > best[0] + 1e-12:
            best = (s, sub)
    assert tuple(idx.tolist()) == best[1]


def test_top_t_float32_comparison_and_forced():
    # two scores that differ only below float32 resolution tie -> lower index
    score = np.array([0.5, 1.0 + 1e-12, 1.0, 0.25])
    assert oracle.select_top_t(score, 1).tolist() == [1]
    assert oracle.select_top_t(score[[0, 2, 1, 3]], 1).tolist() == [1]
    forced = np.array([False, False, False, True])
    assert oracle.select_top_t(score, 2, forced).tolist() == [1, 3]
    with pytest.raises(ValueError):
        oracle.select_top_t(score, 0)


# ------------------------------------------------------------- step 5
def _spd_problem(rng, n, t, mu_eps=0.01, spread=2.0):
    A = np.exp(rng.standard_normal((n, t)) * spread - 3)
    G = A.T @ A
    mu = mu_eps * np.trace(G) / t
    return A, G + mu * np.eye(t), A.sum(0) + mu, mu


@pytest.mark.parametrize("seed", range(8))
def test_nnls_exhaustive_supports(seed):
    """For t <= 9 enumerate every support, keep the unique KKT point, and
    compare with block principal pivoting."""
    rng = np.random.default_rng(100 + seed)
    t = int(rng.integers(2, 10))
    _, Hm, f, _ = _spd_problem(rng, 12, t, mu_eps=float(rng.choice([0.0, 1e-3, 1e-1])) + 1e-9)
    # make some constraints bind: random f with negative parts
    f = f - rng.uniform(0, 1.5, t) * np.abs(f)
    w, _ = oracle.nnls_bpp(Hm, f)
    found = []
    for r in range(t + 1):
        for sup in itertools.combinations(range(t), r):
            x = np.zeros(t)
            if r:
                s = list(sup)
                x[s] = np.linalg.solve(Hm[np.ix_(s, s)], f[s])
            g = Hm @ x - f
            on = np.zeros(t, bool)
            on[list(sup)] = True
            if (x[on] > 0).all() and (g[~on] >= -1e-12).all():
                found.append(x)
    assert len(found) == 1
    np.testing.assert_allclose(w, found[0], rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("seed", range(5))
def test_nnls_matches_scipy_and_kkt(seed):
    """Same minimiser as scipy's Lawson-Hanson on the stacked system
    [A; sqrt(mu) I] w ~ [1; sqrt(mu) 1]; KKT holds."""
    rng = np.random.default_rng(200 + seed)
    n, t = 40, 15
    A = np.exp(rng.standard_normal((n, t)) * 2 - 2)
    w, beta, mu, Hm, f = oracle.fit_beta(A, eps_mu=1e-3)
    ws, _ = scipy_nnls(np.vstack([A, math.sqrt(mu) * np.eye(t)]),
                       np.concatenate([np.ones(n), math.sqrt(mu) * np.ones(t)]), maxiter=10000)
    np.testing.assert_allclose(w, ws, rtol=1e-7, atol=1e-10)
    assert oracle.nnls_kkt_violation(Hm, f, w) < 1e-10
    assert np.all(np.isneginf(beta[w == 0]))
    np.testing.assert_allclose(np.exp(beta[w > 0]), w[w > 0], rtol=1e-14)


def test_nnls_all_negative_gives_zero():
    Hm = np.array([[2.0, 0.5], [0.5, 1.0]])
    w, _ = oracle.nnls_bpp(Hm, np.array([-1.0, -3.0]))
    assert w.tolist() == [0.0, 0.0]


# ------------------------------------------------------------- step 6
def test_values_normal_equation_and_lstsq():
    rng = np.random.default_rng(5)
    n, t, d = 30, 8, 5
    A = np.exp(rng.standard_normal((n, t)))
    w = rng.uniform(0.1, 3, t)
    X = oracle.biased_softmax(A, w)
    np.testing.assert_allclose(X.sum(1), 1.0, rtol=1e-14)
    O, Vs = rng.standard_normal((n, d)), rng.standard_normal((t, d))
    Cv, lam = oracle.fit_values(X, O, Vs, eps_lambda=1e-2)
    lhs = X.T @ (O - X @ Cv)
    np.testing.assert_allclose(lhs, lam * (Cv - Vs), atol=1e-12)
    Cv0, lam0 = oracle.fit_values(X, O, Vs, eps_lambda=0.0)
    assert lam0 == 0.0
    np.testing.assert_allclose(Cv0, np.linalg.lstsq(X, O, rcond=None)[0], rtol=1e-8, atol=1e-10)
    np.testing.assert_allclose(X.T @ (O - X @ Cv0), 0, atol=1e-11)   # residual orthogonal to X


def test_biased_softmax_is_softmax_with_bias():
    """X = rownorm(A' diag w) equals softmax(logits + log w) for any lse shift."""
    rng = np.random.default_rng(6)
    L = rng.standard_normal((4, 5)) * 3
    lse = rng.standard_normal(4)
    w = rng.uniform(0.2, 2, 5)
    X = oracle.biased_softmax(np.exp(L - lse[:, None]), w)
    Z = L + np.log(w)
    E = np.exp(Z - Z.max(1, keepdims=True))
    np.testing.assert_allclose(X, E / E.sum(1, keepdims=True), rtol=1e-13)


# ------------------------------------------------------------- global
@pytest.mark.parametrize("eps", [0.0, 1e-2, 1.0])
def test_t_equals_T_reproduces_cache(eps):
    """With t = T and n >= T: idx = all, w = 1 (beta = 0), C_v = V, and the
    compacted attention equals the full one, for any ridge (it pulls toward
    the same point)."""
    rng = np.random.default_rng(7)
    T, n, d = 24, 48, 6
    K, V = _rand(rng, T, d), _rand(rng, T, d)
    Q = K[rng.integers(0, T, n)] + 0.5 * _rand(rng, n, d)
    r = oracle.compact_head(Q, K, V, T, eps_mu=eps + 1e-12, eps_lambda=eps + 1e-12)
    assert r.idx.tolist() == list(range(T))
    np.testing.assert_allclose(r.w, 1.0, atol=1e-9)
    np.testing.assert_allclose(r.beta, 0.0, atol=1e-9)
    np.testing.assert_allclose(r.Cv, V, atol=1e-7)
    np.testing.assert_allclose(r.mass, 1.0, atol=1e-12)
    Qt = _rand(rng, 9, d)
    np.testing.assert_allclose(oracle.attend(Qt, r.Ck, r.beta, r.Cv, 1 / math.sqrt(d)),
                               oracle.attend_full(Qt, K, V, 1 / math.sqrt(d)), atol=1e-7)


def _golden_q0():
    rows = []
    with open(os.path.join(GOLDEN, "q0_mass.txt")) as fh:
        for line in fh:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


@pytest.mark.parametrize("T,t,full_mass,unbiased", _golden_q0())
def test_page_q0_example(T, t, full_mass, unbiased):
    """The page's q = 0 example: full mass T, unbiased compact mass t; the
    fitted bias restores it.  With every A'_qi = 1/T the ridge problem is
    symmetric, so w_i = (T + eps)/(t + eps) exactly (closed form)."""
    d, n, eps = 4, 10, 1e-2
    rng = np.random.default_rng(T)
    K, V = _rand(rng, T, d), _rand(rng, T, d)
    Q = np.zeros((n, d))
    r = oracle.compact_head(Q, K, V, t, eps_mu=eps, eps_lambda=eps)
    assert np.allclose(np.exp(r.lse), full_mass, rtol=1e-12)
    assert r.idx.tolist() == list(range(t))            # all scores tie -> lowest indices
    assert abs(np.exp(r.lse[0]) * (1.0 / T) * t - unbiased) < 1e-9
    np.testing.assert_allclose(r.w, (T + eps) / (t + eps), rtol=1e-12)
    compact_mass = np.exp(r.beta).sum()                 # sum_i exp(0 + beta_i)
    np.testing.assert_allclose(compact_mass, t * (T + eps) / (t + eps), rtol=1e-12)
    assert abs(compact_mass - full_mass) / full_mass < eps


def test_bf16_rounding_is_nearest_even():
    """The generator's float64 -> bf16 rounding picks the nearest bf16 value
    (ties to even), checked against the two neighbouring bf16 values."""
    from workloads.gen import round_to_bf16_bits
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(4000) * 10, [1 + 2 ** -8, 1 + 3 * 2 ** -8, -1.5]])
    bits = round_to_bf16_bits(x)
    val = oracle.decode(bits, "bf16")
    for xi, vi, bi in zip(x, val, bits):
        up = oracle.decode(np.array([bi + 1], np.uint16), "bf16")[0]
        dn = oracle.decode(np.array([bi - 1], np.uint16), "bf16")[0]
        err = abs(xi - vi)
        assert err <= abs(xi - up) and err <= abs(xi - dn)
        if err == abs(xi - up) or err == abs(xi - dn):
            assert int(bi) % 2 == 0
