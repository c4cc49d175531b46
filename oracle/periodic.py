"""Float64 oracle of periodic compaction ("Thought-Aware KV Cache Compaction"
explainer, section 2 D "Compaction periodique"; "Fast KV Compaction via
Attention Matching" explainer, section 4, "Compaction en ligne": compaction
repeated during decoding keeps reasoning intact).

TEST INFRASTRUCTURE ONLY (see oracle/am.py).

What the page fixes: the compaction runs every P new tokens instead of once,
so the cache holds between t and t + P entries.  Readings taken where it is
silent:

* A compacted cache is (C_k, beta, C_v): a query attends to it with the bias
  beta_i added to the scaled logit of key i and reads C_v.  A period
  compacts the t entries it has (their biases and fp32 values) together
  with the P new tokens (bias 0, their own values): the Attention Matching
  steps run on that cache with the biases in its logits, so the targets
  (mass and outputs of the reference queries) are those of the cache as it
  stands.
* The fit scales the kept entries' existing weights:
  A'_qi = exp(S_q,idx_i + bias_idx_i - lse_q), w' >= 0 by the NNLS with
  ridge mu ||w' - 1||^2, and the new bias is bias_idx_i + log w'_i (-inf
  where w'_i = 0).  The ridge pulls toward "no change" (the kept entries'
  biases as they were), as it pulls toward beta = 0 for a fresh cache, and a
  full budget returns the cache unchanged.
* C_v: least squares against the outputs with ridge lambda ||C_v - V[idx]||^2,
  V[idx] the kept entries' current values.
* Keys are ranked by the RMS of their (biased) attention weights over the
  reference queries, as for a fresh cache.
* The reference queries of each period are an input (the page's are the
  model's own; the synthetic ones come from the workload generator).
"""
from __future__ import annotations

import numpy as np

from .am import (EPS_LAMBDA_DEFAULT, EPS_MU_DEFAULT, HeadResult, key_scores, nnls_bpp, select_top_t)


def attention_biased(Q, K, V, bias, scale: float, row_chunk: int = 1024):
    """Logits S = Q K^T * scale + bias (one bias per key), per-row
    log-sum-exp, outputs O = softmax(S) V, and the column sums of P^2 with
    P = softmax(S).  Keys with bias -inf take no attention."""
    n = Q.shape[0]
    lse = np.empty(n)
    O = np.empty((n, V.shape[1]))
    colsq = np.zeros(K.shape[0])
    for a in range(0, n, row_chunk):
        b = min(n, a + row_chunk)
        S = (Q[a:b] @ K.T) * scale + bias[None, :]
        m = S.max(axis=1)
        lse[a:b] = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
        P = np.exp(S - lse[a:b, None])
        O[a:b] = P @ V
        colsq += (P * P).sum(axis=0)
    return lse, O, colsq


def compact_head_biased(Q, K, V, bias, t: int, *, scale: float | None = None, forced=None,
                        eps_mu: float = EPS_MU_DEFAULT, eps_lambda: float = EPS_LAMBDA_DEFAULT,
                        idx=None) -> HeadResult:
    """One compaction of a cache whose keys carry input biases (float64).

    K [T][d], V [T][d] (the values as the cache holds them), bias [T] (-inf
    allowed).  Returns a HeadResult whose beta is the new bias of each kept
    entry (input bias + log of the fitted weight) and w the fitted weights
    (scales of the kept entries' existing weights).  `idx` (ascending), when
    given, replaces the top-t selection (the fits continued from another
    valid selection)."""
    n, d = Q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    bias = np.asarray(bias, dtype=np.float64)
    lse, O, colsq = attention_biased(Q, K, V, bias, scale)
    score = key_scores(colsq, n)
    if idx is None:
        idx = select_top_t(score, t, forced)
    t = len(idx)
    Ck = K[idx]
    # relative mass of the kept entries, their input biases included
    Ap = np.exp((Q @ Ck.T) * scale + bias[idx][None, :] - lse[:, None])
    G = Ap.T @ Ap
    mu = eps_mu * np.trace(G) / t
    Hm = G + mu * np.eye(t)
    f = Ap.sum(axis=0) + mu
    w, _ = nnls_bpp(Hm, f)
    with np.errstate(divide="ignore"):
        beta = bias[idx] + np.where(w > 0, np.log(np.where(w > 0, w, 1.0)), -np.inf)
    # X_qi = A'_qi w_i / sum_k A'_qk w_k: the compacted cache's attention weights
    num = Ap * w[None, :]
    X = num / num.sum(axis=1, keepdims=True)
    M = X.T @ X
    lam = eps_lambda * np.trace(M) / t
    M = M + lam * np.eye(t)
    R = X.T @ O + lam * V[idx]
    L = np.linalg.cholesky(M)
    Cv = np.linalg.solve(L.T, np.linalg.solve(L, R))
    return HeadResult(idx=idx, score=score, lse=lse, O=O, Ck=Ck, w=w, beta=beta, Cv=Cv, mu=mu, lam=lam,
                      mass=Ap @ w)


def periodic_compaction(K_all, V_all, queries, t: int, T0: int, P: int, *, scale: float | None = None,
                        eps_mu: float = EPS_MU_DEFAULT, eps_lambda: float = EPS_LAMBDA_DEFAULT):
    """A decoding run with compaction every P tokens.

    K_all, V_all: the keys / values of all T0 + k P tokens in order;
    queries(p) -> the reference queries of period p (p = 0 compacts the
    first T0 tokens).  After period p the cache holds t entries: returns the
    list of (positions, C_k, beta, C_v) after each period, positions being
    token indices of K_all."""
    total = K_all.shape[0]
    if T0 < t or (total - T0) % P:
        raise ValueError("the stream must be T0 >= t tokens plus whole periods of P")
    pos = np.arange(T0)
    Ck, Cv = K_all[:T0], V_all[:T0]
    beta = np.zeros(T0)
    out = []
    for p in range(1 + (total - T0) // P):
        if p > 0:
            new = np.arange(T0 + (p - 1) * P, T0 + p * P)
            pos = np.concatenate([pos, new])
            Ck = np.concatenate([Ck, K_all[new]])
            Cv = np.concatenate([Cv, V_all[new]])
            beta = np.concatenate([beta, np.zeros(P)])
        r = compact_head_biased(queries(p), Ck, Cv, beta, t, scale=scale, eps_mu=eps_mu, eps_lambda=eps_lambda)
        pos, Ck, beta, Cv = pos[r.idx], r.Ck, r.beta, r.Cv
        out.append((pos.copy(), Ck.copy(), beta.copy(), Cv.copy()))
    return out
