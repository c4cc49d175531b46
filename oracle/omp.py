"""Float64 oracle of key selection by orthogonal matching pursuit ("Fast KV
Compaction via Attention Matching", section 2 "Pipeline algorithmique", key
selection: keys chosen greedily to best meet the attention-mass objective,
then NNLS for the weights).

TEST INFRASTRUCTURE ONLY (see oracle/am.py).

The page names the method and its objective only.  Readings taken:

* Dictionary and target: the columns p_j of the relative-mass matrix of all T
  keys, P_qj = exp(S_qj - lse_q) (the attention probabilities), against the
  all-ones target -- the same relative-mass objective the NNLS fits.
* Greedy step (plain orthogonal matching pursuit): with S the keys chosen so
  far and r = 1 - P_S w the residual of the least-squares fit of 1 on the
  columns of S (r = 1 while S is empty), pick the key outside S with the
  largest normalised correlation <p_j, r> / ||p_j||; ties go to the lowest
  position; a column of norm 0 is picked only when no other key is left.
* Forced positions start S (ascending); the pursuit fills S up to t.
* The pursuit's own weights are discarded: beta and C_v are then fitted on
  the chosen keys exactly as for the highest-attention selection (ridge NNLS
  and ridge least squares of oracle/am.py).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .am import (EPS_LAMBDA_DEFAULT, EPS_MU_DEFAULT, HeadResult, attention_reference, biased_softmax, fit_beta,
                 fit_values, mass_matrix)


def omp_residual(P: np.ndarray, S) -> np.ndarray:
    """1 - P_S w with w the least-squares fit of 1 on the columns S of P."""
    y = np.ones(P.shape[0])
    if len(S) == 0:
        return y
    A = P[:, list(S)]
    w, *_ = np.linalg.lstsq(A, y, rcond=None)
    return y - A @ w


def omp_select(P: np.ndarray, t: int, forced=None):
    """Greedy pursuit on the columns of P (n x T, non-negative).  Returns
    (order, idx): the chosen positions in the order they were chosen (forced
    ones first, ascending), and the same positions sorted ascending."""
    n, T = P.shape
    if not 1 <= t <= T:
        raise ValueError("budget outside [1, T]")
    norms = np.sqrt((P * P).sum(axis=0))
    S = [int(j) for j in np.flatnonzero(forced)] if forced is not None else []
    if len(S) > t:
        raise ValueError("more forced positions than the budget")
    chosen = np.zeros(T, dtype=bool)
    chosen[S] = True
    while len(S) < t:
        r = omp_residual(P, S)
        corr = np.full(T, -np.inf)
        live = (~chosen) & (norms > 0)
        corr[live] = (P[:, live].T @ r) / norms[live]
        if live.any():
            j = int(np.argmax(corr))                 # first maximum: lowest position
        else:
            j = int(np.flatnonzero(~chosen)[0])      # only zero columns left
        S.append(j)
        chosen[j] = True
    order = np.array(S, dtype=np.int64)
    return order, np.sort(order)


@dataclass
class OmpResult(HeadResult):
    order: np.ndarray = None


def compact_head_omp(Q, K, V, t: int, *, scale: float | None = None, forced=None,
                     eps_mu: float = EPS_MU_DEFAULT, eps_lambda: float = EPS_LAMBDA_DEFAULT,
                     row_chunk: int = 1024) -> OmpResult:
    """One KV head with the keys chosen by the pursuit; every other step as
    in compact_head (float64 inputs)."""
    n, d = Q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    lse, O, _ = attention_reference(Q, K, V, scale, row_chunk)
    P = np.exp((Q @ K.T) * scale - lse[:, None])
    order, idx = omp_select(P, t, forced)
    Ck = K[idx]
    Ap = mass_matrix(Q, Ck, lse, scale)
    w, beta, mu, _, _ = fit_beta(Ap, eps_mu)
    X = biased_softmax(Ap, w)
    Cv, lam = fit_values(X, O, V[idx], eps_lambda)
    norms = np.sqrt((P * P).sum(axis=0))
    return OmpResult(idx=idx, score=norms, lse=lse, O=O, Ck=Ck, w=w, beta=beta, Cv=Cv, mu=mu, lam=lam,
                     mass=Ap @ w, order=order)
