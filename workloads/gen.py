"""Seeded synthetic inputs for KV-cache compaction.

This module only draws numbers: it holds none of the compaction method's
arithmetic, and both the CPU oracle and the GPU path read the bytes it
produces.  Values are drawn in float64 and rounded exactly once to the
storage dtype (round-to-nearest-even), so the two sides see identical inputs.

Recipe per KV head (every draw comes from numpy's PCG64 seeded by
SeedSequence([cfg_id, sequence, layer, kv_head, stream]); stream 0 = cache,
1 = reference queries, 2 = held-out queries, 3 = budgets of the whole call):

* K_pre = G U + noise_k * N(0,1), with G ~ N(0,1) of shape T x r and a basis
  U ~ N(0, 1/r) of shape r x d (so the low-rank part has unit variance).
  Segmented caches draw one (G, U) pair per segment of T/segments tokens.
  The first `sinks` rows are scaled by 4 (attention sinks).
* Per-head temperature: K = s_h * K_pre, s_h ~ U(lo, hi) when the workload
  has a scale range (the reference queries stay unscaled, so s_h acts as an
  inverse softmax temperature).
* V ~ N(0, 1).
* Reference queries: Q = K_pre[j] + N(0, q_noise_var), j uniform in [0, T).
  GQA groups are stacked along the n rows.
* RoPE (when rope_theta is set): half-split rotary pairs (i, i + d/2) with
  frequency theta^(-2i/d); K row i is rotated at position i and a query drawn
  from row j at position T + j (a repeated-prefill reading: the queries come
  from a second copy of the context).
"""
from __future__ import annotations

import numpy as np

from .configs import Workload

STREAM_CACHE, STREAM_QREF, STREAM_TEST, STREAM_BUDGET, STREAM_WINDOW, STREAM_BIAS = 0, 1, 2, 3, 4, 5


def rng_for(w: Workload, h: int, stream: int) -> np.random.Generator:
    s, layer, kv = w.head_address(h)
    return np.random.default_rng(np.random.SeedSequence([w.cfg_id, s, layer, kv, stream]))


# ---------------------------------------------------------------- rounding
def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> bfloat16 bit patterns (uint16), one round-to-nearest-even.

    Works on the float64 bit pattern directly so there is no intermediate
    float32 rounding (which could round twice).  Only zero and normal
    bfloat16 magnitudes are accepted.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    ax = np.abs(x)
    if np.any((ax != 0) & (ax < 2.0 ** -126)) or np.any(ax >= 2.0 ** 127) or not np.all(np.isfinite(x)):
        raise ValueError("value outside the normal bfloat16 range")
    b = x.view(np.uint64)
    drop = np.uint64(45)                       # 52 - 7 mantissa bits dropped
    lsb = (b >> drop) & np.uint64(1)
    r = ((b + (np.uint64(1) << np.uint64(44)) - np.uint64(1) + lsb) >> drop) << drop
    y32 = r.view(np.float64).astype(np.float32)   # exact: y is a bfloat16 value
    return (y32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_to_bf16_bits(x)
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(dtype)


# ---------------------------------------------------------------- rotary
def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Half-split rotary embedding of rows x[i] at positions pos[i] (float64)."""
    d = x.shape[1]
    half = d // 2
    inv = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / d)
    ang = pos.astype(np.float64)[:, None] * inv[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[:, :half], x[:, half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=1)


# ---------------------------------------------------------------- one head
def _rank(w: Workload, layer: int) -> int:
    if w.rank_by_layer is None:
        return w.rank
    lo, hi = w.rank_by_layer
    if w.layers == 1:
        return lo
    return int(round(lo + (hi - lo) * layer / (w.layers - 1)))


def head_cache_f64(w: Workload, h: int) -> tuple[np.ndarray, np.ndarray, np.ndarray, float]:
    """(K_pre, K, V, s_h) in float64, before rounding.  K includes RoPE."""
    rng = rng_for(w, h, STREAM_CACHE)
    _, layer, _ = w.head_address(h)
    s_h = 1.0
    if w.scale_range is not None:
        s_h = float(rng.uniform(*w.scale_range))
    T, d = w.T, w.d
    if w.segments:
        K_pre = np.empty((T, d))
        bounds = np.linspace(0, T, w.segments + 1).astype(np.int64)
        for a, b in zip(bounds[:-1], bounds[1:]):
            G = rng.standard_normal((b - a, w.seg_rank))
            U = rng.standard_normal((w.seg_rank, d)) * np.sqrt(1.0 / w.seg_rank)
            K_pre[a:b] = G @ U
        K_pre += w.noise_k * rng.standard_normal((T, d))
    else:
        r = _rank(w, layer)
        G = rng.standard_normal((T, r))
        U = rng.standard_normal((r, d)) * np.sqrt(1.0 / r)
        K_pre = G @ U + w.noise_k * rng.standard_normal((T, d))
    if w.sinks:
        K_pre[: w.sinks] *= 4.0
    V = rng.standard_normal((T, d))
    K = s_h * K_pre
    if w.rope_theta is not None:
        K = rope(K, np.arange(T), w.rope_theta)
    return K_pre, K, V, s_h


def queries_f64(w: Workload, h: int, K_pre: np.ndarray, count: int, stream: int) -> np.ndarray:
    rng = rng_for(w, h, stream)
    j = rng.integers(0, w.T, size=count)
    Q = K_pre[j] + np.sqrt(w.q_noise_var) * rng.standard_normal((count, w.d))
    if w.rope_theta is not None:
        Q = rope(Q, w.T + j, w.rope_theta)
    return Q


def head_inputs(w: Workload, h: int, with_test: bool = True) -> dict:
    """Storage-dtype inputs of head h: Q [n][d], K [T][d], V [T][d], Qt [n_test][d].

    bf16 arrays are uint16 bit patterns; f32 arrays are float32.
    """
    K_pre, K, V, _ = head_cache_f64(w, h)
    Q = queries_f64(w, h, K_pre, w.n, STREAM_QREF)
    out = {
        "Q": to_storage(Q, w.dtype),
        "K": to_storage(K, w.dtype),
        "V": to_storage(V, w.dtype),
    }
    if with_test:
        out["Qt"] = to_storage(queries_f64(w, h, K_pre, w.n_test, STREAM_TEST), w.dtype)
    return out


# ---------------------------------------------------------------- budgets
def budgets(w: Workload) -> np.ndarray:
    """Per-head budgets t_h (int32 [H]).

    Uniform workloads return t everywhere.  Non-uniform ones read "budgets
    summing to budget_frac * T, Dirichlet(1), floored" as: the mean budget is
    budget_frac * T (total round(budget_frac * T * H)); the forced keeps count
    inside each t_h; the remaining part is a Dirichlet(1) share of what is
    left, floored at budget_floor and capped at n - forced (so that t_h <= n),
    water-filled so the floor and cap keep the total, then rounded by largest
    remainder.
    """
    H = w.H
    if w.t is not None:
        return np.full(H, w.t, dtype=np.int32)
    forced = w.keep_first + w.keep_last
    total = int(round(w.budget_frac * w.T * H))
    rest = total - forced * H
    lo, hi = float(w.budget_floor), float(min(w.n, w.T) - forced)
    if not (lo * H <= rest <= hi * H):
        raise ValueError("budget total infeasible under floor/cap")
    rng = np.random.default_rng(np.random.SeedSequence([w.cfg_id, 0, 0, 0, STREAM_BUDGET]))
    p = rng.dirichlet(np.ones(H))
    # water-fill: find c with sum(clip(c * p, lo, hi)) == rest (monotone in c)
    a, b = 0.0, rest / p.min() + hi
    for _ in range(200):
        c = 0.5 * (a + b)
        if np.clip(c * p, lo, hi).sum() < rest:
            a = c
        else:
            b = c
    x = np.clip(b * p, lo, hi)
    x *= rest / x.sum()
    x = np.clip(x, lo, hi)
    base = np.floor(x).astype(np.int64)
    short = rest - int(base.sum())
    order = np.argsort(-(x - base), kind="stable")
    i = 0
    while short > 0:
        k = order[i % H]
        if base[k] < hi:
            base[k] += 1
            short -= 1
        i += 1
    while short < 0:
        k = order[::-1][i % H]
        if base[k] > lo:
            base[k] -= 1
            short += 1
        i += 1
    out = (base + forced).astype(np.int32)
    assert int(out.sum()) == total
    return out


def forced_mask(w: Workload) -> np.ndarray:
    """Boolean [T]: positions that every head must keep."""
    m = np.zeros(w.T, dtype=bool)
    m[: w.keep_first] = True
    if w.keep_last:
        m[w.T - w.keep_last:] = True
    return m


# ---------------------------------------------------------------- window
def segment_bounds(w: Workload) -> np.ndarray:
    """int32 [S+1]: the segment boundaries the cache was generated with (one
    segment when the workload has none)."""
    if not w.segments:
        return np.array([0, w.T], dtype=np.int32)
    return np.linspace(0, w.T, w.segments + 1).astype(np.int64).astype(np.int32)


def window_queries(w: Workload, h: int, R: int) -> np.ndarray:
    """Storage-dtype [R][d]: queries of the last R tokens of head h (the
    selection window of thought-aware compaction), drawn like the reference
    queries but from positions T - R .. T - 1, rotated at their own positions."""
    K_pre, _, _, _ = head_cache_f64(w, h)
    rng = rng_for(w, h, STREAM_WINDOW)
    j = np.arange(w.T - R, w.T)
    Q = K_pre[j] + np.sqrt(w.q_noise_var) * rng.standard_normal((R, w.d))
    if w.rope_theta is not None:
        Q = rope(Q, j, w.rope_theta)
    return to_storage(Q, w.dtype)



def compacted_cache_extras(w: Workload, h: int, n_old: int, V_f64: np.ndarray, off_frac: float = 0.03):
    """Seeded stand-ins for what an earlier compaction leaves on the first
    n_old positions of head h's cache (periodic compaction: t compacted
    entries followed by new tokens):
      bias  float32 [T]: log of a weight drawn from U(0.3, 4) on the first
            n_old positions, -inf on a share `off_frac` of them (entries an
            earlier fit switched off, never position 0), 0 on the new tokens;
      V     float32 [T][d]: the cache's values with N(0, 0.05^2) added on the
            first n_old positions (refitted values are not bfloat16 numbers),
            unchanged on the new tokens.
    Random numbers only: the values carry no compaction arithmetic."""
    rng = rng_for(w, h, STREAM_BIAS)
    T = V_f64.shape[0]
    bias = np.zeros(T)
    bias[:n_old] = np.log(rng.uniform(0.3, 4.0, n_old))
    off = rng.random(n_old) < off_frac
    off[0] = False
    bias[:n_old][off] = -np.inf
    V = np.array(V_f64, dtype=np.float64)
    V[:n_old] += 0.05 * rng.standard_normal((n_old, V.shape[1]))
    return bias.astype(np.float32), V.astype(np.float32)
