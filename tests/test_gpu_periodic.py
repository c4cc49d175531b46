"""GPU parity of the compaction of a biased cache (kvc_compact_biased, the
step of periodic compaction) against the float64 oracle
(oracle/periodic.py), through the C ABI.

Inputs are seeded: a synthetic cache whose first entries carry the biases and
fp32 values an earlier compaction would leave (workloads.compacted_cache_extras),
or two periods run back to back where the second period's cache is the
oracle's own first-period result rounded to fp32 (no input comes from the
CUDA path).  Tolerances are those of tests/parity.py."""
import math

import numpy as np
import pytest

import oracle
from oracle.periodic import compact_head_biased
from workloads import WORKLOADS, compacted_cache_extras, small_variant
from workloads.batch import generate

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


from parity import compare_head, idx_check, to_torch  # noqa: E402


def _run_gpu(dtype, Q, K, bias, V, Qt, t, params=None):
    """All heads through kvc_compact_biased and kvc_attend.  Q, K, Qt in the
    storage dtype (numpy), bias fp32 [H][T], V fp32 [H][T][d]."""
    import kv_cache_compaction_03_b300 as kvc
    H = Q.shape[0]
    b = torch.full((H,), t, dtype=torch.int32, device="cuda")
    c = kvc.compact_biased_tensors(to_torch(Q, dtype), to_torch(K, dtype),
                                   torch.from_numpy(np.ascontiguousarray(bias, dtype=np.float32)).cuda(),
                                   torch.from_numpy(np.ascontiguousarray(V, dtype=np.float32)).cuda(), b, params)
    Oh, st2 = kvc.attend_tensors(to_torch(Qt, dtype), c)
    torch.cuda.synchronize()
    total = int(c.offsets[-1].item())
    return {
        "status": c.head_status.cpu().numpy(), "attend_status": st2.cpu().numpy(),
        "offsets": c.offsets.cpu().numpy().astype(np.int64), "idx": c.idx.cpu().numpy().astype(np.int64),
        "beta": c.beta.cpu().numpy().astype(np.float64), "Cv": c.C_v.cpu().numpy().astype(np.float64),
        "Ck": c.C_k.float().cpu().numpy().astype(np.float64), "Ohat": Oh.cpu().numpy().astype(np.float64),
        "w": kvc.workspace_view(c, kvc.WS_W, total, torch.float32).cpu().numpy().astype(np.float64),
    }


def _check_heads(g, dtype, Q, K, bias, V, Qt, t, heads=None):
    H = Q.shape[0]
    for h in range(H) if heads is None else heads:
        Qh, Kh, Qth = (oracle.decode(a[h], dtype) for a in (Q, K, Qt))
        bh = bias[h].astype(np.float64)
        Vh = V[h].astype(np.float64)
        r = compact_head_biased(Qh, Kh, Vh, bh, t)
        o0, o1 = g["offsets"][h], g["offsets"][h + 1]
        gi = g["idx"][o0:o1]
        ok, swapped = idx_check(gi, r.idx, r.score)
        assert ok, f"head {h}: kept sets differ beyond the exemption"
        if swapped:
            r = compact_head_biased(Qh, Kh, Vh, bh, t, idx=gi)
        np.testing.assert_array_equal(g["Ck"][o0:o1], Kh[gi])
        Ohat = oracle.attend(Qth, r.Ck, r.beta, r.Cv, 1 / math.sqrt(Qh.shape[1]))
        compare_head(g, h, r, Ohat, {"head": h}, Q=Qh, bias=bh[r.idx])


def _synthetic(w, n_old):
    x = generate(w, workers=1)
    H = w.H
    bias = np.zeros((H, w.T), dtype=np.float32)
    V = np.zeros((H, w.T, w.d), dtype=np.float32)
    for h in range(H):
        bias[h], V[h] = compacted_cache_extras(w, h, n_old, oracle.decode(x["V"][h], w.dtype))
    return x, bias, V


@pytest.mark.parametrize("d", [64, 128])
def test_biased_cache_bf16(d):
    """Compacted entries (biases, some switched off, fp32 values) followed by
    new tokens: several key tiles, ragged tails."""
    w = small_variant(WORKLOADS[2], H=3, n=320, T=1000, t=100, d=d)
    x, bias, V = _synthetic(w, n_old=700)
    g = _run_gpu(w.dtype, x["Q"], x["K"], bias, V, x["Qt"], w.t)
    assert np.all(g["status"] == 0), g["status"]
    assert np.all(g["attend_status"] == 0)
    _check_heads(g, w.dtype, x["Q"], x["K"], bias, V, x["Qt"], w.t)


def test_biased_cache_fp32():
    """The fp32 path (FFMA kernels) with input biases."""
    w = small_variant(WORKLOADS[1], H=2, n=256, T=700, t=64)
    x, bias, V = _synthetic(w, n_old=500)
    g = _run_gpu(w.dtype, x["Q"], x["K"], bias, V, x["Qt"], w.t)
    assert np.all(g["status"] == 0), g["status"]
    _check_heads(g, w.dtype, x["Q"], x["K"], bias, V, x["Qt"], w.t)


def test_full_budget_returns_the_cache():
    """Keeping every entry returns the biases and values unchanged."""
    w = small_variant(WORKLOADS[2], H=2, n=256, T=200, t=200)
    x, bias, V = _synthetic(w, n_old=150)
    g = _run_gpu(w.dtype, x["Q"], x["K"], bias, V, x["Qt"], w.t)
    assert np.all(g["status"] == 0), g["status"]
    for h in range(w.H):
        o0, o1 = g["offsets"][h], g["offsets"][h + 1]
        assert g["idx"][o0:o1].tolist() == list(range(w.T))
        fin = np.isfinite(bias[h])
        assert np.abs(g["beta"][o0:o1][fin] - bias[h][fin]).max() <= 1e-4
        assert np.all(np.isneginf(g["beta"][o0:o1][~fin]))
        assert np.linalg.norm(g["Cv"][o0:o1] - V[h]) / np.linalg.norm(V[h]) <= 1e-3


def test_zero_bias_is_a_fresh_compaction():
    """Biases 0 and the cache's own values (as fp32): the same compaction as
    kvc_compact of the fresh cache."""
    w = small_variant(WORKLOADS[2], H=2, n=320, T=900, t=90)
    x = generate(w, workers=1)
    bias = np.zeros((w.H, w.T), dtype=np.float32)
    V = np.stack([oracle.decode(x["V"][h], w.dtype) for h in range(w.H)]).astype(np.float32)
    g = _run_gpu(w.dtype, x["Q"], x["K"], bias, V, x["Qt"], w.t)
    assert np.all(g["status"] == 0)
    _check_heads(g, w.dtype, x["Q"], x["K"], bias, V, x["Qt"], w.t)
    from parity import run_gpu
    g0, _ = run_gpu(w, inputs=x)
    # the two paths round the logits in another order: near-ties may swap
    for h in range(w.H):
        a = set(g0["idx"][g0["offsets"][h]:g0["offsets"][h + 1]].tolist())
        b = set(g["idx"][g["offsets"][h]:g["offsets"][h + 1]].tolist())
        assert len(a & b) >= 0.98 * w.t, (h, len(a & b))


def test_two_periods_back_to_back():
    """Period 0 compacts T0 tokens (the oracle); period 1 compacts its t
    entries (rounded to fp32) with P new tokens, on the GPU and in the
    oracle, against the next reference queries."""
    w = small_variant(WORKLOADS[2], H=2, n=256, T=768, t=96)
    x = generate(w, workers=1)
    T0, P, t = 512, 256, w.t
    H, d = w.H, w.d
    K1 = np.zeros((H, t + P, d), dtype=x["K"].dtype)
    bias1 = np.zeros((H, t + P), dtype=np.float32)
    V1 = np.zeros((H, t + P, d), dtype=np.float32)
    for h in range(H):
        Qh, Kh, Vh = (oracle.decode(x[k][h], w.dtype) for k in "QKV")
        r0 = oracle.compact_head(Qh, Kh[:T0], Vh[:T0], t)
        K1[h, :t] = x["K"][h][r0.idx]
        K1[h, t:] = x["K"][h][T0:]
        bias1[h, :t] = r0.beta.astype(np.float32)
        V1[h, :t] = r0.Cv.astype(np.float32)
        V1[h, t:] = Vh[T0:].astype(np.float32)
    g = _run_gpu(w.dtype, x["Q"], K1, bias1, V1, x["Qt"], t)
    assert np.all(g["status"] == 0), g["status"]
    _check_heads(g, w.dtype, x["Q"], K1, bias1, V1, x["Qt"], t)


def test_switched_off_head_flagged():
    """A head whose every entry has bias -inf has no attention to match
    (NONFINITE); the other heads are unaffected."""
    import kv_cache_compaction_03_b300 as kvc
    w = small_variant(WORKLOADS[2], H=3, n=256, T=512, t=64)
    x, bias, V = _synthetic(w, n_old=300)
    bias[1, :] = -np.inf
    g = _run_gpu(w.dtype, x["Q"], x["K"], bias, V, x["Qt"], w.t)
    assert g["status"].tolist() == [0, kvc.ERR_NONFINITE, 0], g["status"]
    _check_heads(g, w.dtype, x["Q"], x["K"], bias, V, x["Qt"], w.t, heads=[0, 2])
