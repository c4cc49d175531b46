"""GPU parity of kvc_attend, the read of a compacted cache with a per-key
bias ("Fast KV Compaction via Attention Matching", section 2 objective and
section 5 on use with standard attention kernels), against the float64
oracle: the decode path (n_q <= 16, a cluster of CTAs per head) and the
query-tile path, ragged per-head lengths, -inf biases, and the degenerate
heads (empty range, every bias -inf)."""
import math

import numpy as np
import pytest

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
from parity import to_torch  # noqa: E402
from workloads.gen import round_to_bf16_bits  # noqa: E402

# fp32 logits of magnitude |s| carry |s| * 2^-24 of rounding; with |s| <~ 20
# and fp32 accumulation over up to 10^4 keys the output is good to ~1e-6
# relative; 2e-5 leaves room for the exp2 approximation.
REL = 2e-5


def _case(seed, H, nq, lens, d, dtype, ninf_frac=0.1):
    rng = np.random.default_rng(seed)
    tot = int(sum(lens))
    Q = rng.standard_normal((H, nq, d))
    Ck = rng.standard_normal((tot, d))
    Cv = rng.standard_normal((tot, d)).astype(np.float32)
    beta = rng.normal(0.0, 1.0, tot).astype(np.float32)
    beta[rng.random(tot) < ninf_frac] = -np.inf
    if dtype == "bf16":
        Qs, Cks = round_to_bf16_bits(Q), round_to_bf16_bits(Ck)
    else:
        Qs, Cks = Q.astype(np.float32), Ck.astype(np.float32)
    offsets = np.zeros(H + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(lens)
    for h in range(H):
        if lens[h] > 0:
            beta[offsets[h]] = 0.0              # at least one finite bias per head
    return Qs, Cks, beta, Cv, offsets


def _run(Qs, Cks, beta, Cv, offsets, nq, d, dtype):
    import kv_cache_compaction_03_b300 as kvc
    H = len(offsets) - 1
    Qt = to_torch(Qs, dtype)
    Ckt = to_torch(Cks, dtype)
    bt = torch.from_numpy(beta).cuda()
    Cvt = torch.from_numpy(Cv).cuda()
    off = torch.from_numpy(offsets).cuda()
    O = torch.empty(H, nq, d, dtype=torch.float32, device="cuda")
    st = torch.empty(H, dtype=torch.int32, device="cuda")
    prob = kvc.make_problem(H, nq, 1, d, kvc.DTYPE_BF16 if dtype == "bf16" else kvc.DTYPE_F32, 1)
    assert kvc.attend(prob, Qt, nq, Ckt, bt, Cvt, off, O, st, 0.0) == 0
    torch.cuda.synchronize()
    return O.cpu().numpy().astype(np.float64), st.cpu().numpy()


def _check(seed, H, nq, lens, d, dtype):
    Qs, Cks, beta, Cv, offsets = _case(seed, H, nq, lens, d, dtype)
    O, st = _run(Qs, Cks, beta, Cv, offsets, nq, d, dtype)
    assert np.all(st == 0), st
    scale = 1.0 / math.sqrt(d)
    for h in range(H):
        o0, o1 = offsets[h], offsets[h + 1]
        ref = oracle.attend(oracle.decode(Qs[h], dtype), oracle.decode(Cks[o0:o1], dtype),
                            beta[o0:o1].astype(np.float64), Cv[o0:o1].astype(np.float64), scale)
        rel = np.linalg.norm(O[h] - ref) / np.linalg.norm(ref)
        assert rel <= REL, (h, rel)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("nq", [1, 4, 16])
def test_decode_ragged(dtype, d, nq):
    """The cluster path: lengths from 1 key (seven CTAs of the cluster idle)
    through one ragged tile to thousands of keys per head."""
    _check(1000 + nq, 6, nq, [1, 7, 33, 260, 1000, 4099], d, dtype)


def test_decode_many_heads():
    """160 heads (the four-CTA cluster taken when the heads outnumber the
    SMs), ragged lengths including 1 and 0-to-few keys per cluster CTA."""
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 700, 160)]
    lens[3], lens[77] = 1, 3
    _check(31, 160, 4, lens, 128, "bf16")


def test_query_tile_path_ragged():
    """n_q = 17 and 200 take the query-tile kernel."""
    _check(7, 3, 17, [5, 300, 1100], 128, "bf16")
    _check(8, 2, 200, [64, 777], 64, "f32")


def test_decode_degenerate_heads():
    """An empty range reports BAD_BUDGET; a head whose biases are all -inf
    reports NONFINITE; the other heads are unaffected."""
    Qs, Cks, beta, Cv, offsets = _case(11, 3, 4, [40, 0, 50], 128, "bf16", ninf_frac=0.0)
    beta[40:90] = -np.inf                     # head 2: every bias -inf
    O, st = _run(Qs, Cks, beta, Cv, offsets, 4, 128, "bf16")
    import kv_cache_compaction_03_b300 as kvc
    assert st[0] == 0 and st[1] == kvc.ERR_BAD_BUDGET and st[2] == kvc.ERR_NONFINITE
    ref = oracle.attend(oracle.decode(Qs[0], "bf16"), oracle.decode(Cks[:40], "bf16"), beta[:40].astype(np.float64),
                        Cv[:40].astype(np.float64), 1.0 / math.sqrt(128))
    assert np.linalg.norm(O[0] - ref) / np.linalg.norm(ref) <= REL


def test_decode_matches_query_tile_path():
    """The same heads through both kernels (n_q = 16 vs the first 16 of 17
    queries) agree to fp32 rounding."""
    Qs, Cks, beta, Cv, offsets = _case(21, 4, 17, [90, 500, 2, 1300], 128, "bf16")
    O17, st17 = _run(Qs, Cks, beta, Cv, offsets, 17, 128, "bf16")
    O16, st16 = _run(np.ascontiguousarray(Qs[:, :16]), Cks, beta, Cv, offsets, 16, 128, "bf16")
    assert np.all(st17 == 0) and np.all(st16 == 0)
    np.testing.assert_allclose(O16, O17[:, :16], rtol=0, atol=2e-5 * np.abs(O17).max())
