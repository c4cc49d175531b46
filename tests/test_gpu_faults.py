"""Per-head failure statuses on the GPU, each made to happen by the inputs or
the parameters of an ordinary call (nothing faults, traps or hangs the GPU):

* NNLS_MAXITER: one block-pivoting step on heads whose weights hit w >= 0
  (the oracle's solution has zero weights, so a second step is needed);
* NOT_SPD: the smallest positive eps_lambda makes lambda round to 0 in fp32;
  keys whose weight is 0 then have an all-zero column of X, so M = X^T X has
  an exactly zero row and the factorisation (or the sweep) meets a zero
  pivot;
* TIMEOUT: a wait limit of one microsecond is below the latency of a tile
  load, so the tensor-core kernels give up, wait for the copies and products
  they had issued, release their tensor memory and report the head.

After each, an ordinary call on the same inputs must give correct results:
the context and the library stay usable."""
import numpy as np
import pytest

from workloads import WORKLOADS, small_variant
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


from parity import compare_head, head_queries, run_gpu, run_oracle_head  # noqa: E402


def _oracle_heads(w, x):
    return [run_oracle_head(w, x, h, w.t) for h in range(w.H)]


def _all_heads_match(w, x, refs):
    g, _ = run_gpu(w, inputs=x)
    assert np.all(g["status"] == 0), g["status"]
    for h, (r, Ohat) in enumerate(refs):
        compare_head(g, h, r, Ohat, {"head": h}, Q=head_queries(w, x, h))


def test_nnls_iteration_cap_reported():
    import kv_cache_compaction_03_b300 as kvc
    w = small_variant(WORKLOADS[2], H=2, n=512, T=2048, t=200)
    x = generate(w, workers=1)
    refs = _oracle_heads(w, x)
    # the constraints bind on every head: the unconstrained solution is not the answer
    assert all(int((r.w == 0).sum()) > 0 for r, _ in refs)
    g, _ = run_gpu(w, inputs=x, params=kvc.default_params(nnls_max_iter=1))
    assert g["status"].tolist() == [kvc.ERR_NNLS_MAXITER] * w.H
    _all_heads_match(w, x, refs)


@pytest.mark.parametrize("cholesky", [True, False])
def test_singular_value_system_reported(cholesky):
    import kv_cache_compaction_03_b300 as kvc
    w = small_variant(WORKLOADS[2], H=2, n=128, T=2048, t=300)
    x = generate(w, workers=1)
    refs = _oracle_heads(w, x)
    assert all(int((r.w == 0).sum()) > 0 for r, _ in refs)
    tiny = float(np.finfo(np.float32).smallest_subnormal)
    prm = kvc.default_params(eps_lambda=tiny, flags=kvc.FLAG_CHOLESKY_CV if cholesky else 0)
    assert prm.eps_lambda > 0.0
    g, _ = run_gpu(w, inputs=x, params=prm)
    assert g["status"].tolist() == [kvc.ERR_NOT_SPD] * w.H
    _all_heads_match(w, x, refs)


def test_wait_timeout_reported_and_context_usable():
    import kv_cache_compaction_03_b300 as kvc
    w = small_variant(WORKLOADS[2], H=4, n=512, T=4096, t=200)
    x = generate(w, workers=1)
    refs = _oracle_heads(w, x)
    g, _ = run_gpu(w, inputs=x, params=kvc.default_params(wait_timeout_us=1))
    st = g["status"].tolist()
    assert set(st) <= {kvc.OK, kvc.ERR_TIMEOUT}, st
    assert st.count(kvc.ERR_TIMEOUT) >= 1, st
    # a head that finished under the short limit finished correctly
    for h, (r, Ohat) in enumerate(refs):
        if st[h] == kvc.OK:
            compare_head(g, h, r, Ohat, {"head": h}, Q=head_queries(w, x, h))
    _all_heads_match(w, x, refs)
