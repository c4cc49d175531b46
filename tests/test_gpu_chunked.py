"""GPU parity of chunked compaction ("Fast KV Compaction via Attention
Matching", section 2, "Compaction par blocs") through kvc_compact_chunked:
every chunk against the float64 oracle compacting that chunk alone (same
tolerances as whole-head compaction), the merged indices against
oracle.compact_chunked, and the merged compact cache read by kvc_attend
against the oracle's attention over the merged cache."""
import math

import numpy as np
import pytest

from workloads import WORKLOADS, small_variant

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
from parity import OHAT_REL, compare_head, continue_oracle, idx_check, to_torch  # noqa: E402
from workloads.batch import generate  # noqa: E402


def _forced(T, keep_first, keep_last):
    m = np.zeros(T, dtype=bool)
    m[:keep_first] = True
    if keep_last:
        m[T - keep_last:] = True
    return m


def _check_chunked(w, buds, keep_first=0, keep_last=0):
    import kv_cache_compaction_03_b300 as kvc
    H, C = buds.shape
    T, n, d = w.T, w.n, w.d
    Tc = T // C
    inputs = generate(w)
    Q, K, V, Qt = (to_torch(inputs[k], w.dtype) for k in ("Q", "K", "V", "Qt"))
    b = torch.from_numpy(buds.astype(np.int32)).cuda()
    prm = kvc.default_params(keep_first=keep_first, keep_last=keep_last)
    c = kvc.compact_chunked_tensors(Q, K, V, b, prm)
    Oh, st2 = kvc.attend_tensors(Qt, c)
    torch.cuda.synchronize()
    status = c.head_status.cpu().numpy()
    assert np.all(status == 0), status
    assert np.all(st2.cpu().numpy() == 0)
    total = int(c.offsets[-1].item())
    g = {
        "offsets": c.offsets.cpu().numpy().astype(np.int64),
        "idx": c.idx.cpu().numpy().astype(np.int64),
        "beta": c.beta.cpu().numpy().astype(np.float64),
        "Cv": c.C_v.cpu().numpy().astype(np.float64),
        "Ck": c.C_k.float().cpu().numpy().astype(np.float64),
        "w": kvc.workspace_view(c, kvc.WS_W, total, torch.float32).cpu().numpy().astype(np.float64),
        "O": kvc.workspace_view(c, kvc.WS_O, H * C * n * d, torch.float32).cpu().numpy().reshape(H * C, n, d),
        "lse": kvc.workspace_view(c, kvc.WS_LSE2, H * C * n, torch.float32).cpu().numpy().reshape(H * C, n)
        * math.log(2),
    }
    Ohat = Oh.cpu().numpy().astype(np.float64)
    scale = 1.0 / math.sqrt(d)
    forced = _forced(T, keep_first, keep_last) if (keep_first or keep_last) else None
    for h in range(H):
        Qh = oracle.decode(inputs["Q"][h], w.dtype)
        Kh = oracle.decode(inputs["K"][h], w.dtype)
        Vh = oracle.decode(inputs["V"][h], w.dtype)
        merged = oracle.compact_chunked(Qh, Kh, Vh, buds[h], scale=scale, forced=forced)
        parts, any_swap = [], False
        for ch in range(C):
            gi = h * C + ch
            o0, o1 = g["offsets"][gi], g["offsets"][gi + 1]
            assert o1 - o0 == buds[h, ch]
            sl = slice(ch * Tc, (ch + 1) * Tc)
            fc = None if forced is None else forced[sl]
            r = oracle.compact_head(Qh, Kh[sl], Vh[sl], int(buds[h, ch]), scale=scale, forced=fc)
            # this chunk's reference attention (fp32 round-off bounds as for a head)
            assert np.abs(g["lse"][gi] - r.lse).max() <= 4e-6 * max(1.0, np.abs(r.lse).max())
            assert np.linalg.norm(g["O"][gi] - r.O) / np.linalg.norm(r.O) <= 2e-4
            # kept positions are whole-cache positions inside this chunk
            pos = g["idx"][o0:o1]
            assert np.all((pos >= ch * Tc) & (pos < (ch + 1) * Tc))
            local = pos - ch * Tc
            ok, swapped = idx_check(local, r.idx, r.score)
            assert ok, f"head {h} chunk {ch}: index sets differ beyond the exemption"
            if swapped:
                any_swap = True
                r = continue_oracle(Qh, Kh[sl], Vh[sl], r, local, scale)
            if fc is not None:
                assert set(np.flatnonzero(fc)) <= set(local.tolist())
            np.testing.assert_array_equal(g["Ck"][o0:o1], Kh[pos])
            gc = {"offsets": np.array([0, o1 - o0]), "idx": local, "w": g["w"][o0:o1], "beta": g["beta"][o0:o1],
                  "Cv": g["Cv"][o0:o1]}
            compare_head(gc, 0, r, None, {"head": h, "chunk": ch}, Q=Qh, scale=scale)
            parts.append(r)
        if not any_swap:
            h0, h1 = g["offsets"][h * C], g["offsets"][(h + 1) * C]
            np.testing.assert_array_equal(g["idx"][h0:h1], merged.idx)
        # the merged compact cache, read by kvc_attend on held-out queries
        Ck = np.concatenate([r.Ck for r in parts])
        beta = np.concatenate([r.beta for r in parts])
        Cv = np.concatenate([r.Cv for r in parts])
        Ohat_or = oracle.attend(oracle.decode(inputs["Qt"][h], w.dtype), Ck, beta, Cv, scale)
        rel = np.linalg.norm(Ohat[h] - Ohat_or) / np.linalg.norm(Ohat_or)
        assert rel <= OHAT_REL, (h, rel)


@pytest.mark.parametrize("d", [64, 128])
def test_chunked_bf16_forced(d):
    """Four chunks of 256 per head, uneven budgets, first-4 / last-64 forced
    keeps (which fall in chunks 0 and 3 only)."""
    w = small_variant(WORKLOADS[2], H=2, n=320, T=1024, d=d)
    buds = np.array([[40, 64, 25, 90], [70, 33, 48, 100]])
    _check_chunked(w, buds, keep_first=4, keep_last=64)


def test_chunked_forced_range_spans_chunks():
    """keep_last longer than a chunk: the last chunk is kept whole and the
    chunk before it keeps the remainder of the range."""
    w = small_variant(WORKLOADS[2], H=1, n=512, T=1200)
    buds = np.array([[50, 80, 400]])
    _check_chunked(w, buds, keep_first=0, keep_last=420)


def test_chunked_fp32_single_chunk_matches_compact():
    """chunks = 1 is kvc_compact: identical outputs bit for bit."""
    import kv_cache_compaction_03_b300 as kvc
    w = small_variant(WORKLOADS[1], H=2, n=256, T=640, t=48)
    inputs = generate(w)
    Q, K, V = (to_torch(inputs[k], w.dtype) for k in ("Q", "K", "V"))
    b = torch.full((2,), 48, dtype=torch.int32, device="cuda")
    a = kvc.compact_tensors(Q, K, V, b)
    c = kvc.compact_chunked_tensors(Q, K, V, b.view(2, 1))
    torch.cuda.synchronize()
    for x, y in ((a.idx, c.idx), (a.beta, c.beta), (a.C_v, c.C_v), (a.C_k, c.C_k), (a.head_status, c.head_status)):
        assert torch.equal(x, y)


def test_chunked_fp32_three_chunks():
    w = small_variant(WORKLOADS[1], H=2, n=256, T=960)
    buds = np.array([[30, 64, 41], [64, 20, 50]])
    _check_chunked(w, buds, keep_first=4, keep_last=8)

