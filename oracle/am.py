"""Float64 CPU oracle for Attention Matching KV-cache compaction.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module.  The
GPU library never calls it and shares no code with it.

What it computes follows "Fast KV Compaction via Attention Matching"
(gist.science explainer of arXiv 2602.16284), section 2 "Methodologie":

* "Objectif principal": a compact cache (C_k, beta, C_v) of t < T entries
  should reproduce, for every reference query q, both the attention output
  exp(q K^T) V / sum exp(q K^T) and the attention mass sum exp(q K^T); the
  per-token scalar bias beta lets t keys carry the mass of T keys (the page's
  q = 0 example: mass T against t).
* "Pipeline algorithmique": keys = the original keys with the highest
  attention over the reference queries, aggregated by RMS; beta fitted by
  non-negative least squares (NNLS) to the attention mass; C_v fitted by
  ordinary least squares to the attention outputs given C_k and beta.

Readings taken where the page is silent (each is exercised by a test):

* Logits carry the usual 1/sqrt(d) scale (the page's formulas omit it);
  beta lives in scaled-logit space.
* Mass is matched relative to each query's own mass: row q of the NNLS is
  divided by m_q = sum_j exp(S_qj), i.e. A'_qi = exp(S_q,idx_i - lse_q) with
  target 1.  (Raw exp(S) overflows and would let a few queries dominate.)
* Both fits carry a ridge toward "no change": mu * ||w - 1||^2 with
  mu = eps_mu * tr(A'^T A') / t, and lambda * ||C_v - V[idx]||^2 with
  lambda = eps_lambda * tr(X^T X) / t.  t = T then reproduces the cache
  exactly for any eps, and the problems are strictly convex.
* Key ranking: score_j = sqrt(mean_q P_qj^2), rounded to float32, sorted by
  (score desc, index asc); forced positions rank first; kept indices are
  returned in ascending order.
* w = 0 gives beta = -inf.
* GQA: the query heads of a group are stacked as the n rows of one KV head.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

EPS_MU_DEFAULT = 1e-2
EPS_LAMBDA_DEFAULT = 1e-2


# ------------------------------------------------------------------ inputs
def decode(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage bytes -> float64 (bf16 is held as uint16 bit patterns)."""
    if dtype == "bf16":
        return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


# ------------------------------------------------------------------ step 1
def attention_reference(Q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                        row_chunk: int = 1024):
    """Logits S = Q K^T * scale, per-row log-sum-exp, outputs O = softmax(S) V,
    and the column sums of P^2 (P = softmax(S)) needed by the key score.

    Objective of section 2: the output exp(qK^T)V / sum exp(qK^T) and the mass
    sum exp(qK^T) (here through lse_q = log m_q).  Rows are processed in
    chunks only to bound memory; every row is independent.
    """
    n = Q.shape[0]
    lse = np.empty(n)
    O = np.empty((n, V.shape[1]))
    colsq = np.zeros(K.shape[0])
    for a in range(0, n, row_chunk):
        b = min(n, a + row_chunk)
        S = (Q[a:b] @ K.T) * scale
        m = S.max(axis=1)
        lse[a:b] = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
        P = np.exp(S - lse[a:b, None])
        O[a:b] = P @ V
        colsq += (P * P).sum(axis=0)
    return lse, O, colsq


# ------------------------------------------------------------------ step 2
def key_scores(colsq: np.ndarray, n: int) -> np.ndarray:
    """RMS of each key's attention weight over the n reference queries
    (section 2, key selection "agreges via RMS")."""
    return np.sqrt(colsq / n)


def select_top_t(score: np.ndarray, t: int, forced: np.ndarray | None = None) -> np.ndarray:
    """Indices of the t highest-scoring keys, ascending.

    The comparison is on the float32 value of the score; equal values go to
    the lower index; forced positions rank above every scored key.
    """
    T = score.shape[0]
    if not (1 <= t <= T):
        raise ValueError("budget out of range")
    key = score.astype(np.float32).astype(np.float64)
    if forced is not None:
        if int(forced.sum()) > t:
            raise ValueError("more forced keys than budget")
        key = np.where(forced, np.inf, key)
    order = sorted(range(T), key=lambda j: (-key[j], j))
    return np.array(sorted(order[:t]), dtype=np.int64)


# ------------------------------------------------------------------ step 4
def mass_matrix(Q: np.ndarray, Ck: np.ndarray, lse: np.ndarray, scale: float) -> np.ndarray:
    """A'_qi = exp(q . C_k[i] * scale) / m_q: the kept keys' attention mass
    for query q relative to its full-cache mass m_q = exp(lse_q)."""
    return np.exp((Q @ Ck.T) * scale - lse[:, None])


# ------------------------------------------------------------------ step 5
def nnls_bpp(Hm: np.ndarray, f: np.ndarray, max_iter: int = 1000, tol: float = 0.0):
    """min_{w >= 0} 1/2 w^T H w - f^T w for symmetric positive definite H.

    Block principal pivoting (Judice & Pires 1994; Kim & Park 2011): keep a
    split of the variables into a free set F and a zero set Z, solve the
    equality-constrained problem on F, and swap every variable that breaks
    feasibility (x_F < 0) or optimality (gradient y_Z < 0); when a full swap
    stops reducing the number of violations, fall back to swapping only the
    largest violating index (which guarantees termination).

    Returns (w, iterations).
    """
    t = f.shape[0]
    Z = np.zeros(t, dtype=bool)          # start with every variable free
    best, budget = t + 1, 3
    for it in range(max_iter):
        x = np.zeros(t)
        F = ~Z
        if F.any():
            Fi = np.flatnonzero(F)
            Lf = np.linalg.cholesky(Hm[np.ix_(Fi, Fi)])
            x[Fi] = np.linalg.solve(Lf.T, np.linalg.solve(Lf, f[Fi]))
        y = Hm @ x - f                  # gradient of the objective
        y[F] = 0.0
        bad = (F & (x < -tol)) | (Z & (y < -tol))
        nbad = int(bad.sum())
        if nbad == 0:
            return np.maximum(x, 0.0), it
        if nbad < best:
            best, budget = nbad, 3
            Z ^= bad
        elif budget > 0:
            budget -= 1
            Z ^= bad
        else:
            j = int(np.flatnonzero(bad).max())
            Z[j] = ~Z[j]
    raise RuntimeError("NNLS did not terminate")


def nnls_kkt_violation(Hm: np.ndarray, f: np.ndarray, w: np.ndarray) -> float:
    """Largest violation of the KKT conditions of min 1/2 w'Hw - f'w, w >= 0,
    relative to max|f|: negativity of w, negative gradient on the zero set,
    nonzero gradient on the support."""
    g = Hm @ w - f
    scale = max(1.0, float(np.abs(f).max()))
    v_neg = float(np.maximum(-w, 0).max(initial=0.0))
    on = w > 0
    v_sup = float(np.abs(g[on]).max(initial=0.0))
    v_zero = float(np.maximum(-g[~on], 0).max(initial=0.0))
    return max(v_neg, v_sup, v_zero) / scale


def fit_beta(Ap: np.ndarray, eps_mu: float = EPS_MU_DEFAULT):
    """NNLS for w = exp(beta) >= 0 matching the relative attention mass:
    min_w ||A' w - 1||^2 + mu ||w - 1||^2, mu = eps_mu * tr(A'^T A') / t.

    Returns (w, beta, mu, H, f) with H = A'^T A' + mu I, f = A'^T 1 + mu 1.
    """
    n, t = Ap.shape
    G = Ap.T @ Ap
    b = Ap.sum(axis=0)
    mu = eps_mu * np.trace(G) / t
    Hm = G + mu * np.eye(t)
    f = b + mu
    w, _ = nnls_bpp(Hm, f)
    with np.errstate(divide="ignore"):
        beta = np.where(w > 0, np.log(np.where(w > 0, w, 1.0)), -np.inf)
    return w, beta, mu, Hm, f


# ------------------------------------------------------------------ step 6
def biased_softmax(Ap: np.ndarray, w: np.ndarray) -> np.ndarray:
    """X_qi = A'_qi w_i / sum_k A'_qk w_k, i.e. softmax_i(q.C_k[i]*scale + beta_i):
    the compacted cache's attention weights (section 2 objective, left side
    of the output equation)."""
    num = Ap * w[None, :]
    return num / num.sum(axis=1, keepdims=True)


def fit_values(X: np.ndarray, O: np.ndarray, Vsel: np.ndarray, eps_lambda: float = EPS_LAMBDA_DEFAULT):
    """Least squares for C_v: min ||X C_v - O||^2 + lambda ||C_v - V[idx]||^2,
    lambda = eps_lambda * tr(X^T X) / t, solved through the normal equations
    (X^T X + lambda I) C_v = X^T O + lambda V[idx] with a Cholesky factor."""
    t = X.shape[1]
    M = X.T @ X
    lam = eps_lambda * np.trace(M) / t
    M = M + lam * np.eye(t)
    R = X.T @ O + lam * Vsel
    L = np.linalg.cholesky(M)
    Cv = np.linalg.solve(L.T, np.linalg.solve(L, R))
    return Cv, lam


# ------------------------------------------------------------------ step 7
def attend(Qt: np.ndarray, Ck: np.ndarray, beta: np.ndarray, Cv: np.ndarray, scale: float) -> np.ndarray:
    """softmax(q C_k^T * scale + beta) C_v: the compacted cache read by a
    standard attention kernel with a per-key bias (section 5, integration
    with FlashAttention-style engines)."""
    L = (Qt @ Ck.T) * scale + beta[None, :]
    m = L.max(axis=1, keepdims=True)
    E = np.exp(L - m)
    return (E / E.sum(axis=1, keepdims=True)) @ Cv


def attend_full(Qt: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Uncompacted attention softmax(q K^T * scale) V."""
    L = (Qt @ K.T) * scale
    m = L.max(axis=1, keepdims=True)
    E = np.exp(L - m)
    return (E / E.sum(axis=1, keepdims=True)) @ V


# ------------------------------------------------------------------ one head
@dataclass
class HeadResult:
    idx: np.ndarray
    score: np.ndarray
    lse: np.ndarray
    O: np.ndarray
    Ck: np.ndarray
    w: np.ndarray
    beta: np.ndarray
    Cv: np.ndarray
    mu: float
    lam: float
    mass: np.ndarray      # sum_i w_i A'_qi per reference query (1 = matched)


def compact_head(Q, K, V, t: int, *, scale: float | None = None, forced=None,
                 eps_mu: float = EPS_MU_DEFAULT, eps_lambda: float = EPS_LAMBDA_DEFAULT,
                 row_chunk: int = 1024) -> HeadResult:
    """All steps for one KV head, in the page's order (float64 inputs)."""
    n, d = Q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    lse, O, colsq = attention_reference(Q, K, V, scale, row_chunk)
    score = key_scores(colsq, n)
    idx = select_top_t(score, t, forced)
    Ck = K[idx]
    Ap = mass_matrix(Q, Ck, lse, scale)
    w, beta, mu, _, _ = fit_beta(Ap, eps_mu)
    X = biased_softmax(Ap, w)
    Cv, lam = fit_values(X, O, V[idx], eps_lambda)
    return HeadResult(idx=idx, score=score, lse=lse, O=O, Ck=Ck, w=w, beta=beta, Cv=Cv,
                      mu=mu, lam=lam, mass=Ap @ w)
