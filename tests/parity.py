"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the float64 oracle on the same seeded inputs, and compare them.

Tolerances (float results) and their source:
* selected indices: identical sets, except a swap between two keys whose
  oracle scores differ by less than 1e-6 relative (the stated exemption);
* beta: |beta_gpu - beta_oracle| <= 1e-3 wherever the oracle weight
  w_i >= 1e-6 * max w and beta_i is determined to that tolerance by fp32
  logits.  The second condition is measured, per weight, by re-solving the
  oracle's fit on the relative masses that fp32 logits give (the raw logit
  and the log-mass rounded to float32 as a fp32 pipeline holds them,
  everything else in float64): a weight whose beta that rounding alone moves
  by more than a quarter of the tolerance is not determined by any fp32
  computation of the logits, and is compared as a weight instead,
  |w_gpu - w_oracle| <= 1e-5 * max w.  Where the oracle's w_i < 1e-6 max w,
  the GPU's must be <= 2e-6 max w.  (When the caller passes no queries the
  tolerance applies to every weight above the floor.)
* C_v: relative Frobenius error <= 2e-3 per head;
* compacted attention on held-out queries: relative Frobenius <= 1e-3 per head;
* intermediates (O, lse, scores) against fp32 round-off bounds derived in the
  tests that use them.
When a head's index set differs within the exemption, beta/C_v/outputs are
compared with the oracle continued from the GPU's selection.
"""
from __future__ import annotations

import math

import numpy as np

import oracle
from workloads import budgets as make_budgets, forced_mask
from workloads.batch import generate

IDX_REL_GAP = 1e-6
BETA_ABS = 1e-3
BETA_W_FLOOR = 1e-6
W_FLOOR_GPU = 2e-6
W_ABS_BELOW = 1e-5
FP32_SENS_SHARE = 0.25
CV_REL = 2e-3
OHAT_REL = 1e-3


def to_torch(a, dtype: str, device="cuda"):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def run_gpu(w, inputs=None, buds=None, params=None):
    """All heads of workload w through kvc_compact + kvc_attend in one call each."""
    import torch
    import kv_cache_compaction_03_b300 as kvc
    if inputs is None:
        inputs = generate(w)
    if buds is None:
        buds = make_budgets(w)
    Q = to_torch(inputs["Q"], w.dtype)
    K = to_torch(inputs["K"], w.dtype)
    V = to_torch(inputs["V"], w.dtype)
    Qt = to_torch(inputs["Qt"], w.dtype)
    b = torch.from_numpy(np.asarray(buds, dtype=np.int32)).cuda()
    prm = params or kvc.default_params(keep_first=w.keep_first, keep_last=w.keep_last)
    c = kvc.compact_tensors(Q, K, V, b, prm)
    Oh, st2 = kvc.attend_tensors(Qt, c)
    torch.cuda.synchronize()
    H, n, d, T = w.H, w.n, w.d, w.T
    total = int(c.offsets[-1].item())
    out = {
        "status": c.head_status.cpu().numpy(),
        "attend_status": st2.cpu().numpy(),
        "offsets": c.offsets.cpu().numpy().astype(np.int64),
        "idx": c.idx.cpu().numpy().astype(np.int64),
        "beta": c.beta.cpu().numpy().astype(np.float64),
        "Cv": c.C_v.cpu().numpy().astype(np.float64),
        "Ck": c.C_k.float().cpu().numpy().astype(np.float64),
        "Ohat": Oh.cpu().numpy().astype(np.float64),
        "O": kvc.workspace_view(c, kvc.WS_O, H * n * d, torch.float32).cpu().numpy().reshape(H, n, d),
        "lse": kvc.workspace_view(c, kvc.WS_LSE2, H * n, torch.float32).cpu().numpy().reshape(H, n) * math.log(2),
        "score": kvc.workspace_view(c, kvc.WS_SCORE, H * T, torch.float32).cpu().numpy().reshape(H, T),
        "w": kvc.workspace_view(c, kvc.WS_W, total, torch.float32).cpu().numpy().astype(np.float64),
    }
    return out, inputs


def run_oracle_head(w, inputs, h, t, idx=None, eps_mu=None):
    Q = oracle.decode(inputs["Q"][h], w.dtype)
    K = oracle.decode(inputs["K"][h], w.dtype)
    V = oracle.decode(inputs["V"][h], w.dtype)
    Qt = oracle.decode(inputs["Qt"][h], w.dtype)
    scale = 1.0 / math.sqrt(w.d)
    forced = forced_mask(w) if (w.keep_first or w.keep_last) else None
    mu_kw = {} if eps_mu is None else {"eps_mu": eps_mu}
    r = oracle.compact_head(Q, K, V, t, forced=forced, **mu_kw)
    if idx is not None and not np.array_equal(idx, r.idx):
        r = continue_oracle(Q, K, V, r, idx, scale, eps_mu)
    Ohat = oracle.attend(Qt, r.Ck, r.beta, r.Cv, scale)
    return r, Ohat


def head_queries(w, inputs, h):
    """Float64 reference queries of head h (for compare_head's Q)."""
    return oracle.decode(inputs["Q"][h], w.dtype)


def continue_oracle(Q, K, V, r, idx, scale, eps_mu=None):
    """The oracle's result for one head continued from a given (valid)
    selection idx instead of its own."""
    Ck = K[idx]
    Ap = oracle.mass_matrix(Q, Ck, r.lse, scale)
    wv, beta, mu, _, _ = oracle.fit_beta(Ap) if eps_mu is None else oracle.fit_beta(Ap, eps_mu)
    X = oracle.biased_softmax(Ap, wv)
    Cv, lam = oracle.fit_values(X, r.O, V[idx])
    return oracle.HeadResult(idx=idx, score=r.score, lse=r.lse, O=r.O, Ck=Ck, w=wv, beta=beta, Cv=Cv, mu=mu,
                             lam=lam, mass=Ap @ wv)


def fp32_logit_beta(Q, r, scale, refit=None, bias=None, eps_mu=None):
    """beta of the oracle's fit re-solved on the relative masses that fp32
    logits give: the raw logit q . C_k[i], the log-mass lse_q and the kept
    keys' input biases (in log2 units) rounded to float32, the scaled sum
    rounded once more (one fused multiply-add), everything else in float64.
    refit(A) -> beta replaces the plain NNLS (for fits with pinned weights);
    bias (float64 [t], the kept keys' input biases) is added to the fitted
    log-weights as the biased compaction does."""
    ln2 = math.log(2.0)
    c2 = float(np.float32(scale / ln2))
    S = (Q @ r.Ck.T).astype(np.float32).astype(np.float64)
    lse2 = (r.lse / ln2).astype(np.float32).astype(np.float64)
    b2 = np.zeros(S.shape[1]) if bias is None else (bias / ln2).astype(np.float32).astype(np.float64)
    with np.errstate(invalid="ignore"):
        l2 = (S * c2 + b2[None, :] - lse2[:, None]).astype(np.float32).astype(np.float64)
    A = np.exp2(l2)
    if refit is not None:
        return refit(A)
    beta = (oracle.fit_beta(A) if eps_mu is None else oracle.fit_beta(A, eps_mu))[1]
    return beta if bias is None else bias + beta


def idx_check(gpu_idx, or_idx, or_score):
    """(ok, swapped): sets equal, or every differing pair within the exemption."""
    a, b = set(gpu_idx.tolist()), set(or_idx.tolist())
    if a == b:
        return True, False
    extra, missing = sorted(a - b), sorted(b - a)
    if len(extra) != len(missing):
        return False, True
    key = or_score.astype(np.float32).astype(np.float64)
    lo = min(key[j] for j in missing)          # weakest oracle-kept key
    hi = max(key[j] for j in extra)            # strongest GPU-only key
    ok = abs(lo - hi) <= IDX_REL_GAP * max(abs(lo), abs(hi))
    return ok, True


def compare_head(g, h, r, Ohat_or, report, Q=None, scale=None, refit=None, bias=None, eps_mu=None):
    """Head h of the GPU's outputs g against the oracle's result r (tolerances
    in the module docstring).  Q (float64 reference queries of the head) and
    scale enable the per-weight fp32 determination of beta."""
    off0, off1 = g["offsets"][h], g["offsets"][h + 1]
    gi = g["idx"][off0:off1]
    ok, swapped = idx_check(gi, r.idx, r.score)
    report["idx_swapped"] = swapped
    assert ok, f"head {h}: index sets differ beyond the exemption"
    assert np.all(np.diff(gi) > 0), "indices not ascending"
    wg = g["w"][off0:off1]
    bg = g["beta"][off0:off1]
    wo, bo = r.w, r.beta
    wmax = wo.max()
    live = wo >= BETA_W_FLOOR * wmax
    determined = np.ones_like(live)
    if Q is not None:
        b32 = fp32_logit_beta(Q, r, scale if scale is not None else 1.0 / math.sqrt(Q.shape[1]), refit, bias, eps_mu)
        with np.errstate(invalid="ignore"):
            sens = np.where(np.isfinite(b32) & live, np.abs(b32 - bo), np.inf)
        determined = sens <= FP32_SENS_SHARE * BETA_ABS
    check = live & determined
    db = np.abs(bg[check] - bo[check])
    report["beta_max_abs"] = float(db.max()) if db.size else 0.0
    small = check & (wo < 1e-2 * wmax)
    report["small_weights"] = int(small.sum())
    report["beta_small_max_abs"] = float(np.abs(bg[small] - bo[small]).max()) if small.any() else 0.0
    report["undetermined"] = int((live & ~determined).sum())
    assert np.all(np.isfinite(bg[check])) and report["beta_max_abs"] <= BETA_ABS, f"head {h}: beta {report['beta_max_abs']}"
    und = live & ~determined
    dw = np.abs(wg[und] - wo[und])
    report["w_undetermined_max_abs"] = float(dw.max() / wmax) if dw.size else 0.0
    assert report["w_undetermined_max_abs"] <= W_ABS_BELOW, f"head {h}: weights {report['w_undetermined_max_abs']}"
    report["w_below_floor_max"] = float(wg[~live].max() / wmax) if (~live).any() else 0.0
    assert report["w_below_floor_max"] <= W_FLOOR_GPU, f"head {h}: weights below the floor {report['w_below_floor_max']}"
    # beta = log w (plus the kept key's input bias on a biased cache)
    b_in = np.zeros_like(bg) if bias is None else np.where(np.isfinite(bias), bias, 0.0)
    np.testing.assert_allclose(np.exp(bg[wg > 0] - b_in[wg > 0]), wg[wg > 0], rtol=2e-6)
    assert np.all(np.isneginf(bg[wg == 0]))
    cv = g["Cv"][off0:off1]
    report["cv_rel"] = float(np.linalg.norm(cv - r.Cv) / np.linalg.norm(r.Cv))
    assert report["cv_rel"] <= CV_REL, f"head {h}: C_v rel {report['cv_rel']}"
    if Ohat_or is not None:
        report["ohat_rel"] = float(np.linalg.norm(g["Ohat"][h] - Ohat_or) / np.linalg.norm(Ohat_or))
        assert report["ohat_rel"] <= OHAT_REL, f"head {h}: held-out rel {report['ohat_rel']}"
    return report
