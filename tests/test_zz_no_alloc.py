"""kvc_compact_noalloc against kvc_compact, through the C ABI.

Some callers cannot allocate device memory. Examples: an engine whose
allocator has reserved the device up front, a latency-critical path where
cudaMalloc would synchronise the device, or a C program with no device
allocator. kvc_compact_noalloc serves them from a fixed device array inside
the library. This file checks three things:
- two calls in a row give the same compaction as kvc_compact on
  caller-allocated workspace, within the parity tolerances of the other tests;
- the second call does not depend on what the first one left in the shared
  array;
- a problem too large for the array is refused before anything is enqueued.

The file name sorts last, so a run that stops at its first failure has
already run every other test.
"""
import numpy as np
import pytest

from parity import BETA_ABS, BETA_W_FLOOR, CV_REL, W_ABS_BELOW, to_torch
from workloads import WORKLOADS, small_variant
from workloads.batch import generate

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_compaction_03_b300 import build
    build.build()
    import kv_cache_compaction_03_b300 as k
    k.lib()
    return k


def _outputs(total, d, dtype, H):
    return (torch.empty(total, dtype=torch.int32, device="cuda"),
            torch.empty(total, d, dtype=dtype, device="cuda"),
            torch.empty(total, dtype=torch.float32, device="cuda"),
            torch.empty(total, d, dtype=torch.float32, device="cuda"),
            torch.empty(H, dtype=torch.int32, device="cuda"))


def test_noalloc_matches_workspace_entry_point_twice(kvc):
    w = small_variant(WORKLOADS[2], H=3, n=320, T=1000, t=100)
    x = generate(w, workers=1)
    Q, K, V = (to_torch(x[k], w.dtype) for k in "QKV")
    b = torch.full((w.H,), w.t, dtype=torch.int32, device="cuda")
    ref = kvc.compact_tensors(Q, K, V, b)
    torch.cuda.synchronize()
    assert ref.head_status.cpu().tolist() == [0] * w.H
    total = int(ref.offsets[-1].item())
    prob = kvc.make_problem(w.H, w.n, w.T, w.d, kvc.DTYPE_BF16, w.t)
    assert kvc.workspace_size(prob) <= kvc.NOALLOC_SCRATCH_BYTES
    r_beta = ref.beta.cpu().numpy().astype(np.float64)
    r_w = np.exp(r_beta)
    r_cv = ref.C_v.cpu().numpy().astype(np.float64)
    for call in range(2):
        idx, Ck, beta, Cv, st = _outputs(total, w.d, Q.dtype, w.H)
        rc = kvc.compact_noalloc(prob, None, Q, K, V, b, ref.offsets, idx, Ck, beta, Cv, st)
        assert rc == 0, kvc.status_string(rc)
        torch.cuda.synchronize()
        assert st.cpu().tolist() == [0] * w.H, call
        assert torch.equal(idx, ref.idx), call
        assert torch.equal(Ck, ref.C_k), call
        g_beta = beta.cpu().numpy().astype(np.float64)
        g_cv = Cv.cpu().numpy().astype(np.float64)
        for h in range(w.H):
            sl = slice(h * w.t, (h + 1) * w.t)
            big = r_w[sl] >= BETA_W_FLOOR * r_w[sl].max()
            assert np.abs(g_beta[sl][big] - r_beta[sl][big]).max() <= BETA_ABS
            assert np.abs(np.exp(g_beta[sl][~big]) - r_w[sl][~big]).max(initial=0.0) <= W_ABS_BELOW * r_w[sl].max()
            rel = np.linalg.norm(g_cv[sl] - r_cv[sl]) / np.linalg.norm(r_cv[sl])
            assert rel <= CV_REL, (call, h, rel)


def test_noalloc_refuses_problems_beyond_its_array(kvc):
    prob = kvc.make_problem(256, 8192, 32768, 128, kvc.DTYPE_BF16, 655)
    assert kvc.workspace_size(prob) > kvc.NOALLOC_SCRATCH_BYTES
    p = 0x100000   # never dereferenced: the call is refused on the host
    rc = kvc.compact_noalloc(prob, None, p, p, p, p, p, p, p, p, p, p)
    assert rc == kvc.ERR_NOALLOC_LIMIT
    assert "scratch" in kvc.status_string(rc)
    timed = kvc.default_params(flags=kvc.FLAG_STAGE_TIMING)
    small = kvc.make_problem(1, 16, 64, 64, kvc.DTYPE_BF16, 8)
    assert kvc.compact_noalloc(small, timed, p, p, p, p, p, p, p, p, p, p) == kvc.ERR_INVALID_ARG
