"""Float64 oracle of the thought-aware compaction planner and fits ("Thought-
Aware KV Cache Compaction" explainer, section 2: B adaptive budget
allocation, C pivot-token protection; built on Attention Matching).

TEST INFRASTRUCTURE ONLY (see oracle/am.py).

What the page fixes: a segment's importance w_i is the mean attention mass
it receives from a selection window (the queries of the last R tokens); the
kept keys of segment i number t_i proportional to sqrt(w_i) * n_i (n_i its
size); tokens whose window attention is consistently above delta = c * mean
attention are pivots, kept exactly with zero bias, and the remaining budget
is shared among the non-pivot tokens.  Readings taken where it is silent:

* alpha_j = mean over the window queries of softmax_j(q K^T * scale); a
  pivot has alpha_j > c * mean_j alpha_j (strictly); w_i = sum of alpha over
  the segment (its mean received mass).
* The budget t counts the pivots; t - #pivots is shared by
  t_i ~ sqrt(w_i) * n_i with n_i the segment's non-pivot count, capped at
  n_i (the excess is re-shared among the uncapped segments, repeatedly), and
  made integral by largest remainder (ties to the lower segment).
* Inside a segment the t_i non-pivot keys are chosen as Attention Matching
  chooses keys (highest RMS attention over the reference queries, float32
  key, ties to the lower position).
* The fits are Attention Matching's with the pivots held at w = 1 (beta = 0)
  and C_v = V: the NNLS and the least squares run over the other kept keys,
  the pivots' mass and output moved to the targets; the ridges mu and lambda
  keep their definitions over all t kept keys.
* Segment boundaries are an input (the page finds them in the text, by
  paragraph breaks).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .am import (EPS_LAMBDA_DEFAULT, EPS_MU_DEFAULT, HeadResult, attention_reference, biased_softmax, key_scores,
                 mass_matrix, nnls_bpp)


def window_attention(Qw: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """alpha_j: the attention key j receives, averaged over the window queries."""
    S = (Qw @ K.T) * scale
    S = S - S.max(axis=1, keepdims=True)
    E = np.exp(S)
    return (E / E.sum(axis=1, keepdims=True)).mean(axis=0)


def detect_pivots(alpha: np.ndarray, c: float) -> np.ndarray:
    """Boolean [T]: alpha_j > c * mean(alpha)."""
    return alpha > c * alpha.mean()


def allocate_budgets(weights, sizes, total: int) -> np.ndarray:
    """Integer t_i ~ sqrt(w_i) * n_i with sum t_i = total and 0 <= t_i <= n_i."""
    w = np.asarray(weights, dtype=np.float64)
    n = np.asarray(sizes, dtype=np.int64)
    if total < 0 or total > int(n.sum()):
        raise ValueError("budget outside [0, sum of segment sizes]")
    share = np.sqrt(np.maximum(w, 0.0)) * n
    x = np.zeros(len(n))
    capped = np.zeros(len(n), dtype=bool)
    left = float(total)
    while True:
        free = ~capped & (share > 0)
        tot = share[free].sum()
        x[free] = left * share[free] / tot if tot > 0 else 0.0
        over = free & (x > n)
        if not over.any():
            break
        x[over] = n[over]
        capped |= over
        left = total - x[capped].sum()
    base = np.minimum(np.floor(x + 1e-12).astype(np.int64), n)
    short = total - int(base.sum())
    frac = x - base
    # largest remainder among the segments with room left, ties to the lower index
    cand = sorted((i for i in range(len(n)) if base[i] < n[i]), key=lambda i: (-frac[i], i))
    for i in cand[:short]:
        base[i] += 1
    short = total - int(base.sum())
    for i in range(len(n)):                      # only if every share was 0: fill in order
        if short == 0:
            break
        add = min(short, int(n[i] - base[i]))
        base[i] += add
        short -= add
    return base


def select_segments(score: np.ndarray, bounds, budgets, pivots: np.ndarray) -> np.ndarray:
    """Per segment [bounds[i], bounds[i+1]): its pivots and its budgets[i]
    non-pivot keys of largest float32 score (ties to the lower position).
    Returns every kept position, ascending."""
    key = score.astype(np.float32).astype(np.float64)
    out = []
    for i in range(len(bounds) - 1):
        lo, hi = int(bounds[i]), int(bounds[i + 1])
        seg = np.arange(lo, hi)
        out.extend(seg[pivots[lo:hi]].tolist())
        cand = [j for j in seg if not pivots[j]]
        cand.sort(key=lambda j: (-key[j], j))
        out.extend(cand[:int(budgets[i])])
    return np.array(sorted(out), dtype=np.int64)


def fit_beta_fixed(Ap: np.ndarray, piv: np.ndarray, eps_mu: float = EPS_MU_DEFAULT):
    """NNLS for the non-pivot weights with the pivots held at w = 1:
    min ||A'_np w + A'_p 1 - 1||^2 + mu ||w - 1||^2 over w >= 0,
    mu = eps_mu * tr(A'^T A') / t over all t kept keys."""
    n, t = Ap.shape
    mu = eps_mu * float((Ap * Ap).sum()) / t
    w = np.ones(t)
    free = ~piv
    if free.any():
        A = Ap[:, free]
        target = 1.0 - Ap[:, piv].sum(axis=1)
        Hm = A.T @ A + mu * np.eye(A.shape[1])
        f = A.T @ target + mu
        w[free], _ = nnls_bpp(Hm, f)
    with np.errstate(divide="ignore"):
        beta = np.where(w > 0, np.log(np.where(w > 0, w, 1.0)), -np.inf)
    return w, beta, mu


def fit_values_fixed(X: np.ndarray, O: np.ndarray, Vsel: np.ndarray, piv: np.ndarray,
                     eps_lambda: float = EPS_LAMBDA_DEFAULT):
    """C_v for the non-pivot rows with the pivot rows held at V:
    min ||X_np C + X_p V_p - O||^2 + lambda ||C - V_np||^2,
    lambda = eps_lambda * tr(X^T X) / t over all t kept keys."""
    t = X.shape[1]
    lam = eps_lambda * float((X * X).sum()) / t
    Cv = Vsel.copy()
    free = ~piv
    if free.any():
        A = X[:, free]
        M = A.T @ A + lam * np.eye(A.shape[1])
        R = A.T @ (O - X[:, piv] @ Vsel[piv]) + lam * Vsel[free]
        L = np.linalg.cholesky(M)
        Cv[free] = np.linalg.solve(L.T, np.linalg.solve(L, R))
    return Cv, lam


@dataclass
class TamResult(HeadResult):
    alpha: np.ndarray = None
    pivots: np.ndarray = None       # boolean [T]
    seg_budgets: np.ndarray = None  # non-pivot keys kept per segment


def plan_head(Qw, K, bounds, t: int, c: float, scale: float):
    """(alpha, pivots, segment budgets) for one head."""
    alpha = window_attention(Qw, K, scale)
    piv = detect_pivots(alpha, c)
    npiv = int(piv.sum())
    if npiv > t:
        raise ValueError("more pivots than the budget")
    S = len(bounds) - 1
    w = np.array([alpha[bounds[i]:bounds[i + 1]].sum() for i in range(S)])
    sizes = np.array([int((~piv[bounds[i]:bounds[i + 1]]).sum()) for i in range(S)])
    return alpha, piv, allocate_budgets(w, sizes, t - npiv)


def compact_head_tam(Q, K, V, Qw, bounds, t: int, c: float, *, scale: float | None = None,
                     eps_mu: float = EPS_MU_DEFAULT, eps_lambda: float = EPS_LAMBDA_DEFAULT, plan=None) -> TamResult:
    """One head: plan (unless given as (alpha, pivots, budgets)), per-segment
    selection, then the fits with the pivots held exactly."""
    n, d = Q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    alpha, piv, bud = plan if plan is not None else plan_head(Qw, K, bounds, t, c, scale)
    lse, O, colsq = attention_reference(Q, K, V, scale)
    score = key_scores(colsq, n)
    idx = select_segments(score, bounds, bud, piv)
    Ck = K[idx]
    Ap = mass_matrix(Q, Ck, lse, scale)
    pk = piv[idx]
    w, beta, mu = fit_beta_fixed(Ap, pk, eps_mu)
    X = biased_softmax(Ap, w)
    Cv, lam = fit_values_fixed(X, O, V[idx], pk, eps_lambda)
    return TamResult(idx=idx, score=score, lse=lse, O=O, Ck=Ck, w=w, beta=beta, Cv=Cv, mu=mu, lam=lam,
                     mass=Ap @ w, alpha=alpha, pivots=piv, seg_budgets=bud)
