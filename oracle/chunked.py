"""Float64 oracle of chunked compaction ("Fast KV Compaction via Attention
Matching", section 2, "Compaction par blocs"): the cache of one KV head is
split into contiguous chunks, each chunk is compacted on its own against the
same reference queries, and the compacted chunks are concatenated.

TEST INFRASTRUCTURE ONLY (see oracle/am.py).
"""
from __future__ import annotations

import numpy as np

from .am import EPS_LAMBDA_DEFAULT, EPS_MU_DEFAULT, HeadResult, compact_head


def compact_chunked(Q, K, V, budgets, *, scale=None, forced=None, eps_mu: float = EPS_MU_DEFAULT,
                    eps_lambda: float = EPS_LAMBDA_DEFAULT) -> HeadResult:
    """Compact K, V (T rows) as len(budgets) equal contiguous chunks with
    budgets[c] kept entries each, then merge: idx are positions in the full
    cache, C_k, beta, C_v are the chunks' results in chunk order.  `forced`
    (boolean [T]) is split with the chunks.  In the merged HeadResult, lse and
    O are the full cache's (recombined from the chunks), score holds the
    chunks' own key scores, mu / lam are chunk 0's, and mass is the merged
    compact cache's mass relative to the full cache's."""
    T = K.shape[0]
    C = len(budgets)
    if C < 1 or T % C:
        raise ValueError("the cache length must be a multiple of the chunk count")
    Tc = T // C
    parts = []
    for c in range(C):
        sl = slice(c * Tc, (c + 1) * Tc)
        fc = None if forced is None else forced[sl]
        parts.append(compact_head(Q, K[sl], V[sl], int(budgets[c]), scale=scale, forced=fc, eps_mu=eps_mu,
                                  eps_lambda=eps_lambda))
    cat = np.concatenate
    # Attention over concatenated blocks decomposes by mass: the full cache's
    # log-mass is the log-sum-exp of the chunks' and its output is their
    # mass-weighted mean; the merged compact cache's relative mass likewise.
    L = np.stack([r.lse for r in parts])
    top = L.max(axis=0)
    wt = np.exp(L - top)
    tot = wt.sum(axis=0)
    lse = top + np.log(tot)
    O = sum(wt[c][:, None] * r.O for c, r in enumerate(parts)) / tot[:, None]
    mass = sum(wt[c] * r.mass for c, r in enumerate(parts)) / tot
    return HeadResult(idx=cat([r.idx + c * Tc for c, r in enumerate(parts)]),
                      score=cat([r.score for r in parts]), lse=lse, O=O,
                      Ck=cat([r.Ck for r in parts]), w=cat([r.w for r in parts]), beta=cat([r.beta for r in parts]),
                      Cv=cat([r.Cv for r in parts]), mu=parts[0].mu, lam=parts[0].lam, mass=mass)
