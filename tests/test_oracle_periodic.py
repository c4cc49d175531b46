"""Pins of the periodic-compaction oracle (oracle/periodic.py) against facts
that do not come from it: the plain Attention Matching oracle, a key bias
written out as repeated keys, the full-budget identity, and the
reparametrisation invariance of the weight fit."""
import math

import numpy as np
import pytest

import oracle
from oracle.periodic import attention_biased, compact_head_biased, periodic_compaction


def _head(seed, n=96, T=160, d=16):
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 0.5, (6, d))
    K = rng.normal(0, 1, (T, 6)) @ U + 0.3 * rng.normal(0, 1, (T, d))
    K[:2] *= 3.0
    V = rng.normal(0, 1, (T, d))
    Q = K[rng.integers(0, T, n)] + rng.normal(0, math.sqrt(0.5), (n, d))
    return Q, K, V


def test_zero_bias_is_attention_matching():
    """With every bias 0 (a fresh cache) one period is the plain compaction."""
    Q, K, V = _head(1)
    a = compact_head_biased(Q, K, V, np.zeros(K.shape[0]), 24)
    b = oracle.compact_head(Q, K, V, 24)
    np.testing.assert_array_equal(a.idx, b.idx)
    np.testing.assert_allclose(a.lse, b.lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(a.w, b.w, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(a.Cv, b.Cv, rtol=1e-9, atol=1e-10)


def test_bias_acts_as_repeated_keys():
    """A bias log m on a key attends exactly like m copies of that key (the
    page's q = 0 argument: mass is counted per key).  Written out as an
    unbiased cache with the repeats, lse and outputs must agree, and each
    copy's RMS score is 1/m of the biased key's."""
    Q, K, V = _head(2, T=40)
    reps = {3: 3, 11: 2, 30: 5}
    bias = np.zeros(K.shape[0])
    rows = []
    for j in range(K.shape[0]):
        m = reps.get(j, 1)
        bias[j] = math.log(m)
        rows += [j] * m
    scale = 1 / math.sqrt(K.shape[1])
    lse_b, O_b, colsq_b = attention_biased(Q, K, V, bias, scale)
    Kr, Vr = K[rows], V[rows]
    L = (Q @ Kr.T) * scale
    mx = L.max(axis=1, keepdims=True)
    E = np.exp(L - mx)
    lse_r = mx[:, 0] + np.log(E.sum(axis=1))
    O_r = (E / E.sum(axis=1, keepdims=True)) @ Vr
    np.testing.assert_allclose(lse_b, lse_r, rtol=0, atol=1e-12)
    np.testing.assert_allclose(O_b, O_r, rtol=0, atol=1e-12)
    P_r = np.exp(L - lse_r[:, None])
    first = {j: rows.index(j) for j in reps}
    for j, m in reps.items():
        np.testing.assert_allclose(math.sqrt(colsq_b[j]) / m, math.sqrt((P_r[:, first[j]] ** 2).sum()), rtol=1e-12)


@pytest.mark.parametrize("seed", [3, 4])
def test_full_budget_returns_the_cache(seed):
    """Keeping every entry: the weights' optimum is w' = 1 (zero residual,
    zero ridge), so the biases come back unchanged and C_v = V."""
    Q, K, V = _head(seed, n=64, T=50)
    rng = np.random.default_rng(seed + 10)
    bias = rng.normal(0, 1.5, K.shape[0])
    bias[7] = -np.inf                      # an entry an earlier fit switched off
    r = compact_head_biased(Q, K, V, bias, K.shape[0])
    np.testing.assert_array_equal(r.idx, np.arange(K.shape[0]))
    fin = np.isfinite(bias)
    np.testing.assert_allclose(r.beta[fin], bias[fin], rtol=0, atol=1e-9)
    assert np.isneginf(r.beta[7])
    np.testing.assert_allclose(r.Cv, V, rtol=0, atol=1e-9)


def test_total_bias_independent_of_its_split():
    """Without the ridge, w -> w / m_i is a reparametrisation: fitting the
    kept entries' weights on top of input biases gives the same total bias as
    fitting them from scratch on the same kept keys (scipy-free check against
    the plain fit of oracle.am on the unbiased relative masses)."""
    Q, K, V = _head(5, n=200, T=120)
    rng = np.random.default_rng(6)
    bias = rng.normal(0, 0.7, K.shape[0])
    eps = 1e-12
    r = compact_head_biased(Q, K, V, bias, 20, eps_mu=eps)
    scale = 1 / math.sqrt(K.shape[1])
    A0 = np.exp((Q @ K[r.idx].T) * scale - r.lse[:, None])        # unbiased, same lse
    w0, beta0, *_ = oracle.fit_beta(A0, eps_mu=eps)
    on = w0 > 1e-6 * w0.max()
    np.testing.assert_array_equal(on, r.w > 1e-6 * r.w.max())
    np.testing.assert_allclose(r.beta[on], beta0[on], rtol=0, atol=1e-6)


def test_periodic_run_shapes_and_first_period():
    """Every period leaves t entries at increasing positions of the stream;
    period 0 is the plain compaction of the first T0 tokens; later periods
    keep only positions seen so far."""
    Q, K, V = _head(7, n=80, T=200)
    t, T0, P = 30, 80, 40
    qs = [Q[:, :] + 0.1 * i for i in range(4)]
    out = periodic_compaction(K, V, lambda p: qs[p], t, T0, P)
    assert len(out) == 1 + (K.shape[0] - T0) // P
    for p, (pos, Ck, beta, Cv) in enumerate(out):
        assert len(pos) == t and np.all(np.diff(pos) > 0)
        assert pos.max() < T0 + p * P
        np.testing.assert_array_equal(Ck, K[pos])
    r0 = oracle.compact_head(qs[0], K[:T0], V[:T0], t)
    np.testing.assert_array_equal(out[0][0], r0.idx)
    np.testing.assert_allclose(out[0][2], r0.beta, rtol=0, atol=1e-9)
