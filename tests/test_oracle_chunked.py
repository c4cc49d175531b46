"""Pins of the chunked-compaction oracle ("Fast KV Compaction via Attention
Matching", section 2, "Compaction par blocs") against facts that do not come
from it: one chunk is the plain compaction; keeping every key of every chunk
reproduces the full cache exactly; the recombined log-mass and output are
the full cache's (closed form of attention over concatenated blocks); the
merged cache's attention is the mass-weighted mean of the chunks'."""
import math

import numpy as np
import pytest

import oracle


def _head(seed, T=48, n=40, d=6):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((T, d)) * 1.5
    V = rng.standard_normal((T, d))
    Q = K[rng.integers(0, T, n)] + 0.5 * rng.standard_normal((n, d))
    return Q, K, V


def test_one_chunk_is_plain_compaction():
    Q, K, V = _head(1)
    a = oracle.compact_chunked(Q, K, V, [12])
    b = oracle.compact_head(Q, K, V, 12)
    assert a.idx.tolist() == b.idx.tolist()
    np.testing.assert_array_equal(a.beta, b.beta)
    np.testing.assert_array_equal(a.Cv, b.Cv)


def test_full_budget_chunks_reproduce_the_cache():
    Q, K, V = _head(2, T=48, n=60)
    r = oracle.compact_chunked(Q, K, V, [16, 16, 16])
    assert r.idx.tolist() == list(range(48))
    np.testing.assert_allclose(r.beta, 0.0, atol=1e-9)
    np.testing.assert_allclose(r.Cv, V, atol=1e-7)
    Qt = np.random.default_rng(3).standard_normal((7, 6))
    s = 1 / math.sqrt(6)
    np.testing.assert_allclose(oracle.attend(Qt, r.Ck, r.beta, r.Cv, s), oracle.attend_full(Qt, K, V, s), atol=1e-7)


def test_recombined_lse_and_output_are_the_full_caches():
    Q, K, V = _head(4, T=60)
    r = oracle.compact_chunked(Q, K, V, [5, 5, 5, 5])
    lse, O, _ = oracle.attention_reference(Q, K, V, 1 / math.sqrt(6))
    np.testing.assert_allclose(r.lse, lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r.O, O, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_merged_attention_is_mass_weighted_mean_of_chunks(seed):
    """softmax over the merged cache = sum_c M_c O_c / sum_c M_c with M_c, O_c
    the chunk caches' own masses and outputs (brute force per query)."""
    Q, K, V = _head(10 + seed, T=40)
    r = oracle.compact_chunked(Q, K, V, [6, 9])
    s = 1 / math.sqrt(6)
    Qt = np.random.default_rng(seed).standard_normal((5, 6))
    got = oracle.attend(Qt, r.Ck, r.beta, r.Cv, s)
    for q in range(5):
        num = np.zeros(6)
        den = 0.0
        for lo, hi in ((0, 6), (6, 15)):
            logits = [float(Qt[q] @ r.Ck[i]) * s + r.beta[i] for i in range(lo, hi)]
            m = sum(math.exp(x) for x in logits)
            o = sum(math.exp(x) / m * r.Cv[i] for x, i in zip(logits, range(lo, hi)))
            num += m * o
            den += m
        np.testing.assert_allclose(got[q], num / den, rtol=1e-10)


def test_forced_positions_follow_their_chunk():
    Q, K, V = _head(5, T=40)
    forced = np.zeros(40, bool)
    forced[[0, 1, 39]] = True
    r = oracle.compact_chunked(Q, K, V, [4, 4], forced=forced)
    assert {0, 1, 39} <= set(r.idx.tolist())


def test_rejects_uneven_chunks():
    Q, K, V = _head(6, T=40)
    with pytest.raises(ValueError):
        oracle.compact_chunked(Q, K, V, [4, 4, 4])
