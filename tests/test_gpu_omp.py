"""GPU parity of key selection by orthogonal matching pursuit
(KVC_FLAG_SELECT_OMP; "Fast KV Compaction via Attention Matching", section 2
"Pipeline algorithmique", key selection) against the float64 oracle.

A greedy pursuit is a chain of argmax decisions, so one near-tie decided
differently by fp32 and fp64 changes every later step.  The test therefore
replays the GPU's own choices in the oracle: every forced position must come
first, and at every later step the GPU's key must be a valid argmax of the
oracle's normalised correlation with the least-squares residual of the keys
chosen before it (within fp32 accuracy: 1e-4 of ||r||).  The fits that follow
are then compared with the oracle continued from the GPU's keys, with the
usual tolerances."""
import math

import numpy as np
import pytest

from workloads import WORKLOADS, budgets, forced_mask, small_variant

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
from oracle.omp import omp_residual  # noqa: E402
from parity import compare_head, continue_oracle, to_torch  # noqa: E402
from workloads.batch import generate  # noqa: E402

CORR_TOL = 1e-4


def _check(w, buds=None):
    import kv_cache_compaction_03_b300 as kvc
    buds = budgets(w) if buds is None else np.asarray(buds)
    inputs = generate(w)
    Q, K, V, Qt = (to_torch(inputs[k], w.dtype) for k in ("Q", "K", "V", "Qt"))
    b = torch.from_numpy(buds.astype(np.int32)).cuda()
    prm = kvc.default_params(keep_first=w.keep_first, keep_last=w.keep_last, flags=kvc.FLAG_SELECT_OMP)
    c = kvc.compact_tensors(Q, K, V, b, prm)
    Oh, st2 = kvc.attend_tensors(Qt, c)
    torch.cuda.synchronize()
    H, mt = w.H, int(buds.max())
    status = c.head_status.cpu().numpy()
    assert np.all(status == 0), status
    assert np.all(st2.cpu().numpy() == 0)
    total = int(c.offsets[-1].item())
    order = kvc.workspace_view(c, kvc.WS_ORDER, H * mt, torch.int32).cpu().numpy().reshape(H, mt)
    g = {"offsets": c.offsets.cpu().numpy().astype(np.int64), "idx": c.idx.cpu().numpy().astype(np.int64),
         "beta": c.beta.cpu().numpy().astype(np.float64), "Cv": c.C_v.cpu().numpy().astype(np.float64),
         "w": kvc.workspace_view(c, kvc.WS_W, total, torch.float32).cpu().numpy().astype(np.float64),
         "Ohat": Oh.cpu().numpy().astype(np.float64)}
    scale = 1.0 / math.sqrt(w.d)
    forced = forced_mask(w) if (w.keep_first or w.keep_last) else None
    exact = 0
    for h in range(H):
        t = int(buds[h])
        Qh = oracle.decode(inputs["Q"][h], w.dtype)
        Kh = oracle.decode(inputs["K"][h], w.dtype)
        Vh = oracle.decode(inputs["V"][h], w.dtype)
        lse, O, _ = oracle.attention_reference(Qh, Kh, Vh, scale)
        P = np.exp(Qh @ Kh.T * scale - lse[:, None])
        norms = np.sqrt((P * P).sum(axis=0))
        og = order[h, :t].astype(np.int64)
        assert len(set(og.tolist())) == t
        nf = 0 if forced is None else int(forced.sum())
        if nf:
            assert og[:nf].tolist() == np.flatnonzero(forced).tolist()
        for s in range(nf, t):
            r = omp_residual(P, og[:s])
            corr = (P.T @ r) / np.where(norms > 0, norms, np.inf)
            corr[og[:s]] = -np.inf
            best = corr.max()
            assert corr[og[s]] >= best - CORR_TOL * np.linalg.norm(r), (h, s, corr[og[s]], best)
            exact += int(corr[og[s]] == best)
        o0, o1 = g["offsets"][h], g["offsets"][h + 1]
        assert g["idx"][o0:o1].tolist() == sorted(og.tolist())
        stub = oracle.HeadResult(idx=np.sort(og), score=norms, lse=lse, O=O, Ck=None, w=None, beta=None, Cv=None,
                                 mu=0.0, lam=0.0, mass=None)
        r_or = continue_oracle(Qh, Kh, Vh, stub, np.sort(og), scale)
        Ohat = oracle.attend(oracle.decode(inputs["Qt"][h], w.dtype), r_or.Ck, r_or.beta, r_or.Cv, scale)
        compare_head(g, h, r_or, Ohat, {"head": h}, Q=Qh, scale=scale)
    return exact


@pytest.mark.parametrize("d", [64, 128])
def test_omp_bf16(d):
    w = small_variant(WORKLOADS[2], H=2, n=256, T=520, t=40, d=d)
    exact = _check(w)
    assert exact >= 0.9 * 2 * 40           # near-ties aside, the GPU takes the oracle's argmax


def test_omp_fp32_tiny_config():
    _check(small_variant(WORKLOADS[1], H=2, n=256, T=700, t=48))


def test_omp_forced_and_nonuniform_budgets():
    """First 4 and last 64 positions forced; per-head budgets differ."""
    w = small_variant(WORKLOADS[4], H=3, n=256, T=640)
    _check(w, buds=[80, 100, 71])
