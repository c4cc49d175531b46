"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs.  Small workloads span several tiles with ragged tails
and cover the degenerate cases; the full-size workloads run every head in one
call (the launch configuration the benchmark times) and compare a sample of
heads that the oracle computes one by one."""
import math

import numpy as np
import pytest

from workloads import WORKLOADS, budgets, small_variant

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


def _check(w, heads=None, buds=None, check_intermediates=True):
    g, inputs = run_gpu(w, buds=buds)
    buds = budgets(w) if buds is None else buds
    assert np.all(g["status"] == 0), g["status"]
    assert np.all(g["attend_status"] == 0)
    heads = range(w.H) if heads is None else heads
    reports = []
    for h in heads:
        r, Ohat = run_oracle_head(w, inputs, h, int(buds[h]))
        if check_intermediates:
            # fp32 logits of magnitude |S| carry ~|S| * 2^-22 of round-off
            smax = np.abs(r.lse).max()
            tol_lse = 4e-6 * max(1.0, smax)
            assert np.abs(g["lse"][h] - r.lse).max() <= tol_lse
            # fp32 arithmetic (bf16 inputs: P enters P V as two bf16 terms,
            # ~2^-17 relative, below fp32 accumulation error)
            o_rel = np.linalg.norm(g["O"][h] - r.O) / np.linalg.norm(r.O)
            assert o_rel <= 2e-4, o_rel
            sc_rel = np.abs(g["score"][h] - r.score) / np.maximum(r.score, 1e-30)
            assert np.quantile(sc_rel, 0.999) <= 1e-4 and sc_rel.max() <= 1e-3
        # C_k is an exact copy of the kept rows
        o0, o1 = g["offsets"][h], g["offsets"][h + 1]
        from oracle import decode
        K = decode(inputs["K"][h], w.dtype)
        np.testing.assert_array_equal(g["Ck"][o0:o1], K[g["idx"][o0:o1]])
        rep = compare_head(g, h, r, Ohat, {"head": h}, Q=head_queries(w, inputs, h))
        reports.append(rep)
    return reports


@pytest.mark.parametrize("d", [64, 128])
def test_small_bf16_ragged(d):
    w = small_variant(WORKLOADS[2], H=3, n=320, T=1000, t=100, d=d)
    _check(w)


def test_small_cholesky_cv_path():
    """C_v through the blocked Cholesky and triangular solves (the
    KVC_FLAG_CHOLESKY_CV alternative to the explicit inverse)."""
    import kv_cache_compaction_03_b300 as kvc
    w = small_variant(WORKLOADS[2], H=2, n=320, T=1000, t=150)
    g, inputs = run_gpu(w, params=kvc.default_params(flags=kvc.FLAG_CHOLESKY_CV))
    assert np.all(g["status"] == 0)
    for h in range(w.H):
        r, Ohat = run_oracle_head(w, inputs, h, w.t)
        compare_head(g, h, r, Ohat, {"head": h}, Q=head_queries(w, inputs, h))


def test_config1_fp32_full():
    _check(WORKLOADS[1])


def test_small_square_t_equals_n():
    w = small_variant(WORKLOADS[5], H=2, n=256, T=700, t=256)
    _check(w)


def test_small_forced_nonuniform_budgets():
    w = small_variant(WORKLOADS[4], H=6, n=512, T=2048)
    buds = budgets(w)
    assert buds.min() >= 100 and buds.max() <= 512 and len(set(buds.tolist())) > 1
    reps = _check(w, buds=buds)
    assert len(reps) == 6


def test_t_equals_T_identity():
    """t = T, n >= T: every key kept, beta = 0, C_v = V, compacted == full."""
    w = small_variant(WORKLOADS[2], H=2, n=256, T=128, t=128)
    g, inputs = run_gpu(w)
    from oracle import decode
    for h in range(w.H):
        o0, o1 = g["offsets"][h], g["offsets"][h + 1]
        assert g["idx"][o0:o1].tolist() == list(range(128))
        assert np.abs(g["beta"][o0:o1]).max() < 1e-4
        V = decode(inputs["V"][h], w.dtype)
        assert np.linalg.norm(g["Cv"][o0:o1] - V) / np.linalg.norm(V) < 1e-3


def test_largest_budget():
    """The solver size limit: t = 4096 kept keys (64 sweep blocks per matrix),
    n = 4096 queries, a cache of 4100 keys (ragged tails everywhere)."""
    w = small_variant(WORKLOADS[2], H=1, n=4096, T=4100, t=4096)
    _check(w, check_intermediates=False)


def test_many_heads():
    """1000 small heads in one call (grids of 1000 in y); a sample of them
    against the oracle."""
    w = small_variant(WORKLOADS[2], H=1000, n=64, T=200, t=24, d=64)
    _check(w, heads=[0, 1, 499, 998, 999], check_intermediates=True)


def test_degenerate_tiny_shapes():
    """A single key, a budget of one, one query, t = T: every output (kept
    keys, beta, C_v, held-out attention) against the oracle."""
    for (n, T, t) in [(5, 1, 1), (3, 70, 1), (1, 64, 2), (7, 65, 65)]:
        w = small_variant(WORKLOADS[2], H=2, n=n, T=T, t=t, d=64)
        g, inputs = run_gpu(w)
        assert np.all(g["status"] == 0), (n, T, t, g["status"])
        assert np.all(g["attend_status"] == 0), (n, T, t)
        for h in range(w.H):
            r, Ohat = run_oracle_head(w, inputs, h, t)
            compare_head(g, h, r, Ohat, {"head": h}, Q=head_queries(w, inputs, h))


def test_bad_budgets_flagged_per_head():
    import kv_cache_compaction_03_b300 as kvc
    w = small_variant(WORKLOADS[2], H=3, n=64, T=256, t=16, d=64)
    from workloads.batch import generate
    from parity import to_torch
    x = generate(w)
    Q, K, V = (to_torch(x[k], w.dtype) for k in "QKV")
    b = torch.tensor([16, 300, 16], dtype=torch.int32, device="cuda")   # head 1 exceeds T
    offsets = torch.tensor([0, 16, 32, 48], dtype=torch.int32, device="cuda")
    prob = kvc.make_problem(3, 64, 256, 64, kvc.DTYPE_BF16, 16)
    prm = kvc.default_params()
    ws = torch.empty(kvc.workspace_size(prob, prm), dtype=torch.uint8, device="cuda")
    idx = torch.empty(48, dtype=torch.int32, device="cuda")
    Ck = torch.empty(48, 64, dtype=torch.bfloat16, device="cuda")
    beta = torch.empty(48, dtype=torch.float32, device="cuda")
    Cv = torch.empty(48, 64, dtype=torch.float32, device="cuda")
    st = torch.empty(3, dtype=torch.int32, device="cuda")
    rc = kvc.compact(prob, prm, Q, K, V, b, offsets, idx, Ck, beta, Cv, st, ws, ws.numel())
    assert rc == 0
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, kvc.ERR_BAD_BUDGET, 0]


def test_nonfinite_input_flagged():
    import kv_cache_compaction_03_b300 as kvc
    w = small_variant(WORKLOADS[2], H=2, n=64, T=256, t=16, d=64)
    from workloads.batch import generate
    from parity import to_torch
    x = generate(w)
    Q, K, V = (to_torch(x[k], w.dtype) for k in "QKV")
    K[1, 7, 3] = float("nan")
    c = kvc.compact_tensors(Q, K, V, torch.full((2,), 16, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    st = c.head_status.cpu().tolist()
    assert st[0] == 0 and st[1] == kvc.ERR_NONFINITE


def test_values_beyond_fp16_range():
    """V of one head scaled by 2^20 (max |V| ~ 5e6, past the fp16 range of
    the attention's P V operand) and of another by 2^-20 (max |V| ~ 5e-6,
    fp16 subnormals): the pass rewrites both heads' values under a power-of-
    two scale, and both match the oracle like an unscaled head."""
    from oracle import decode
    from workloads.batch import generate
    from workloads.gen import round_to_bf16_bits
    w = small_variant(WORKLOADS[2], H=3, n=320, T=1000, t=100)
    x = generate(w, workers=1)
    for h, f in ((1, 2.0 ** 20), (2, 2.0 ** -20)):
        x["V"][h] = round_to_bf16_bits(decode(x["V"][h], w.dtype) * f)
    g, inputs = run_gpu(w, inputs=x)
    assert np.all(g["status"] == 0), g["status"]
    buds = budgets(w)
    for h in range(w.H):
        r, Ohat = run_oracle_head(w, inputs, h, int(buds[h]))
        o_rel = np.linalg.norm(g["O"][h] - r.O) / np.linalg.norm(r.O)
        assert o_rel <= 2e-4, (h, o_rel)
        compare_head(g, h, r, Ohat, {"head": h}, Q=head_queries(w, inputs, h))


@pytest.mark.parametrize("cfg,sample", [(2, None), (5, [0, 37, 77, 127]), (4, [0, 55, 111]), (3, [0, 131, 255])])
def test_full_config_sampled_heads(cfg, sample):
    w = WORKLOADS[cfg]
    reps = _check(w, heads=sample, check_intermediates=True)
    print({cfg: [(r["head"], round(r["beta_max_abs"], 6), round(r["cv_rel"], 6), round(r["ohat_rel"], 6))
                 for r in reps]})
