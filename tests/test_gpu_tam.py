"""GPU parity of thought-aware compaction (kvc_compact_tam; "Thought-Aware KV
Cache Compaction" explainer, section 2: segment budgets t_i ~ sqrt(w_i) n_i,
pivot tokens kept exactly) against the float64 oracle.

The plan is integer decisions taken from floating point (a threshold, a
largest-remainder rounding), so it is compared where it is unique: pivots
except keys within 1e-5 of the threshold, budgets exactly unless the
rounding has a near-tie (then only its invariants).  The rest is compared
with the oracle continued from the GPU's plan: the kept positions (with the
usual near-tie exemption), beta = 0 and C_v = V exactly on the pivots, and
the usual tolerances elsewhere."""
import math

import numpy as np
import pytest

from workloads import WORKLOADS, segment_bounds, small_variant, window_queries

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_compaction_03_b300 import build
    build.build()
    import kv_cache_compaction_03_b300 as kvc
    kvc.lib()


import oracle  # noqa: E402
from oracle.tam import allocate_budgets, compact_head_tam, fit_beta_fixed, window_attention  # noqa: E402
from parity import compare_head, to_torch  # noqa: E402
from workloads.batch import generate  # noqa: E402


def _check(w, buds, R, c):
    import kv_cache_compaction_03_b300 as kvc
    inputs = generate(w)
    Q, K, V, Qt = (to_torch(inputs[k], w.dtype) for k in ("Q", "K", "V", "Qt"))
    win = np.stack([window_queries(w, h, R) for h in range(w.H)])
    Qw = to_torch(win, w.dtype)
    bounds = segment_bounds(w)
    bt = torch.from_numpy(bounds).cuda()
    b = torch.from_numpy(np.asarray(buds, dtype=np.int32)).cuda()
    cmp, segb, piv = kvc.compact_tam_tensors(Q, K, V, Qw, bt, b, c)
    Oh, st2 = kvc.attend_tensors(Qt, cmp)
    torch.cuda.synchronize()
    status = cmp.head_status.cpu().numpy()
    assert np.all(status == 0), status
    assert np.all(st2.cpu().numpy() == 0)
    total = int(cmp.offsets[-1].item())
    g = {"offsets": cmp.offsets.cpu().numpy().astype(np.int64), "idx": cmp.idx.cpu().numpy().astype(np.int64),
         "beta": cmp.beta.cpu().numpy().astype(np.float64), "Cv": cmp.C_v.cpu().numpy().astype(np.float64),
         "w": kvc.workspace_view(cmp, kvc.WS_W, total, torch.float32).cpu().numpy().astype(np.float64),
         "Ohat": Oh.cpu().numpy().astype(np.float64)}
    segb = segb.cpu().numpy()
    piv = piv.cpu().numpy().astype(bool)
    scale = 1.0 / math.sqrt(w.d)
    S = len(bounds) - 1
    n_piv_total = 0
    for h in range(w.H):
        Qh = oracle.decode(inputs["Q"][h], w.dtype)
        Kh = oracle.decode(inputs["K"][h], w.dtype)
        Vh = oracle.decode(inputs["V"][h], w.dtype)
        Qwh = oracle.decode(win[h], w.dtype)
        alpha = window_attention(Qwh, Kh, scale)
        delta = c * alpha.mean()
        near = np.abs(alpha - delta) <= 1e-5 * delta
        assert np.array_equal(piv[h][~near], (alpha > delta)[~near])
        n_piv_total += int(piv[h].sum())
        # budgets from the GPU's pivots
        wts = np.array([alpha[bounds[i]:bounds[i + 1]].sum() for i in range(S)])
        sizes = np.array([int((~piv[h][bounds[i]:bounds[i + 1]]).sum()) for i in range(S)])
        left = int(buds[h]) - int(piv[h].sum())
        want = allocate_budgets(wts, sizes, left)
        assert int(segb[h].sum()) == left and np.all(segb[h] <= sizes) and np.all(segb[h] >= 0)
        share = np.sqrt(wts) * sizes
        fr = left * share / share.sum() - np.floor(left * share / share.sum())
        if np.sort(np.abs(np.subtract.outer(fr, fr))[np.triu_indices(S, 1)])[:1].min(initial=1.0) > 1e-9:
            assert segb[h].tolist() == want.tolist(), (h, segb[h], want)
        # the rest, continued from the GPU's plan
        r = compact_head_tam(Qh, Kh, Vh, Qwh, bounds, int(buds[h]), c, plan=(alpha, piv[h], segb[h]))
        o0, o1 = g["offsets"][h], g["offsets"][h + 1]
        kept_piv = piv[h][g["idx"][o0:o1]]
        assert np.all(g["beta"][o0:o1][kept_piv] == 0.0)
        np.testing.assert_array_equal(g["Cv"][o0:o1][kept_piv], Vh[g["idx"][o0:o1][kept_piv]])
        assert set(np.flatnonzero(piv[h])) <= set(g["idx"][o0:o1].tolist())
        Ohat = oracle.attend(oracle.decode(inputs["Qt"][h], w.dtype), r.Ck, r.beta, r.Cv, scale)
        kp = piv[h][r.idx]
        compare_head(g, h, r, Ohat, {"head": h}, Q=Qh, scale=scale, refit=lambda A, kp=kp: fit_beta_fixed(A, kp)[1])
    return n_piv_total


def test_tam_reasoning_trace_segments():
    """The reasoning-trace cache (segments, no forced keys): 16 segments of 64
    keys, a window of the last 32 tokens, per-head budgets."""
    w = small_variant(WORKLOADS[4], H=3, n=256, T=1024)
    npiv = _check(w, [120, 160, 100], R=32, c=3.0)
    assert npiv > 0


def test_tam_bf16_d64_no_pivots_one_budget_each():
    """A threshold no key reaches: no pivots, budgets by weight alone."""
    w = small_variant(WORKLOADS[4], H=2, n=192, T=768, d=64)
    assert _check(w, [90, 77], R=16, c=1e6) == 0


def test_tam_bf16_window_on_tensor_cores():
    """A window of 128 queries takes the tensor-core attention pass."""
    w = small_variant(WORKLOADS[4], H=2, n=256, T=1024)
    _check(w, [150, 130], R=128, c=8.0)


def test_tam_fp32():
    w = small_variant(WORKLOADS[4], H=2, n=128, T=512, dtype="f32")
    _check(w, [60, 64], R=16, c=2.0)
