"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/kvc.h declares, sizes workspaces, and rejects bad
arguments before it touches the device."""
import ctypes
import os
import re

import pytest

import kv_cache_compaction_03_b300 as kvc
from kv_cache_compaction_03_b300 import build as kbuild
from workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    kbuild.build()
    return kvc.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "kvc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol():
    names = _declared()
    assert len(names) >= 7
    L = kvc.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(kvc.EXPORTS)


def test_version_and_status_strings():
    assert "sm_103a" in kvc.version()
    for code in (0, 1, 2, 3, 4, 5, 16, 17, 18, 19, 20, 21):
        assert kvc.status_string(code) not in ("", "unknown status")
    assert kvc.status_string(12345) == "unknown status"


def test_default_params():
    p = kvc.default_params()
    assert p.scale == 0.0 and abs(p.eps_mu - 1e-2) < 1e-9 and abs(p.eps_lambda - 1e-2) < 1e-9
    assert p.nnls_max_iter >= 8 and p.refine_iters >= 1 and p.flags == 0


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_workspace_sizes(cfg):
    w = WORKLOADS[cfg]
    from workloads import budgets
    mt = int(budgets(w).max())
    prob = kvc.make_problem(w.H, w.n, w.T, w.d, kvc.DTYPE_BF16 if w.dtype == "bf16" else kvc.DTYPE_F32, mt)
    ws = kvc.workspace_size(prob, kvc.default_params(keep_first=w.keep_first, keep_last=w.keep_last))
    # must hold at least the fp32 reference outputs, scores and the mass matrix
    lower = 4 * w.H * (w.n * w.d + w.T + w.n * mt)
    assert ws >= lower
    assert ws < 64 * 2 ** 30           # fits easily in HBM
    for item in range(5):
        off = kvc.workspace_offset(prob, None, item)
        assert off % 256 == 0 and off < ws


def _call(prob, prm=None, ws_bytes=1 << 20, ptr=0x100000, **over):
    args = dict(Q=ptr, K=ptr, V=ptr, budgets=ptr, offsets=ptr, idx=ptr, Ck=ptr, beta=ptr, Cv=ptr, status=ptr,
                ws=ptr)
    args.update(over)
    return kvc.compact(prob, prm, args["Q"], args["K"], args["V"], args["budgets"], args["offsets"], args["idx"],
                       args["Ck"], args["beta"], args["Cv"], args["status"], args["ws"], ws_bytes, stream=0)


def test_rejects_bad_problems_on_host():
    good = kvc.make_problem(2, 64, 256, 128, kvc.DTYPE_BF16, 32)
    bad = [
        kvc.make_problem(0, 64, 256, 128, 0, 32),      # no heads
        kvc.make_problem(2, 0, 256, 128, 0, 32),       # no queries
        kvc.make_problem(2, 64, 256, 96, 0, 32),       # unsupported d
        kvc.make_problem(2, 64, 256, 128, 7, 32),      # unknown dtype
        kvc.make_problem(2, 64, 256, 128, 0, 300),     # max_t > T
        kvc.make_problem(2, 64, 8192, 128, 0, 5000),   # max_t above the solver limit
        kvc.make_problem(2, 64, 256, 128, 0, 0),
    ]
    for p in bad:
        assert _call(p) == kvc.ERR_INVALID_ARG
    assert _call(good, ptr=0x100000, Q=None) == kvc.ERR_INVALID_ARG
    assert _call(good, Q=0x100004) == kvc.ERR_ALIGN
    assert _call(good, ws_bytes=16) == kvc.ERR_WORKSPACE
    assert _call(good, prm=kvc.default_params(eps_mu=0.0)) == kvc.ERR_INVALID_ARG
    assert _call(good, prm=kvc.default_params(flags=8)) == kvc.ERR_INVALID_ARG
    assert _call(good, prm=kvc.default_params(keep_first=200, keep_last=100)) == kvc.ERR_INVALID_ARG
    assert _call(good, prm=kvc.default_params(wait_timeout_us=0)) == kvc.ERR_INVALID_ARG


def test_chunked_rejects_bad_shapes_on_host():
    ok = kvc.make_problem(2, 64, 1000, 64, kvc.DTYPE_BF16, 250)
    # the workspace of 4 chunks is that of the per-chunk problem
    assert kvc.workspace_size_chunked(ok, None, 4) == kvc.workspace_size(
        kvc.make_problem(8, 64, 250, 64, kvc.DTYPE_BF16, 250))
    assert kvc.workspace_size_chunked(ok, None, 1) == kvc.workspace_size(
        kvc.make_problem(2, 64, 1000, 64, kvc.DTYPE_BF16, 250))
    bad = [
        (kvc.make_problem(2, 64, 1000, 64, 0, 100), 3),      # 1000 % 3 != 0
        (kvc.make_problem(2, 64, 1000, 64, 0, 300), 4),      # max_t > T / chunks
        (kvc.make_problem(2, 64, 1000, 64, 0, 100), 0),      # no chunks
        (kvc.make_problem(40000, 64, 1000, 64, 0, 100), 2),  # H * chunks above the grid limit
    ]
    for p, c in bad:
        with pytest.raises(kvc.KvcError):
            kvc.workspace_size_chunked(p, None, c)
        ptr = 0x100000
        assert kvc.compact_chunked(p, None, c, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1 << 30,
                                   stream=0) == kvc.ERR_INVALID_ARG
    # forced keeps count positions of the whole cache, not of one chunk
    prm = kvc.default_params(keep_first=4, keep_last=400)
    assert kvc.workspace_size_chunked(ok, prm, 4) > 0
    ptr = 0x100000
    assert kvc.compact_chunked(ok, None, 4, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 16,
                               stream=0) == kvc.ERR_WORKSPACE
    assert kvc.compact_chunked(ok, None, 4, 0x100004, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1 << 30,
                               stream=0) == kvc.ERR_ALIGN
    assert _call(kvc.make_problem(70000, 64, 256, 64, 0, 32)) == kvc.ERR_INVALID_ARG   # H above the grid limit


def test_attend_rejects_bad_args_on_host():
    p = kvc.make_problem(2, 1, 1, 128, kvc.DTYPE_BF16, 1)
    assert kvc.attend(p, 0x1000, 0, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0.0, 0) == kvc.ERR_INVALID_ARG
    assert kvc.attend(p, 0x1008, 4, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0.0, 0) == kvc.ERR_ALIGN
    assert kvc.attend(p, 0x1000, 4, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, -1.0, 0) == kvc.ERR_INVALID_ARG


def test_struct_layouts_match_header():
    assert ctypes.sizeof(kvc.Problem) == 24
    assert ctypes.sizeof(kvc.Params) == 40
    assert ctypes.sizeof(kvc.HeadRecord) == 32


def test_biased_rejects_bad_args_on_host():
    p = kvc.make_problem(2, 64, 256, 128, kvc.DTYPE_BF16, 32)
    ws = kvc.workspace_size_biased(p)
    assert ws > kvc.workspace_size(p)          # room for the key biases
    ptr = 0x100000

    def call(prm=None, bias=ptr, V=ptr, ws_bytes=ws):
        return kvc.compact_biased(p, prm, ptr, ptr, bias, V, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ws_bytes,
                                  stream=0)
    assert call(bias=None) == kvc.ERR_INVALID_ARG
    assert call(bias=0x100002) == kvc.ERR_ALIGN
    assert call(V=0x100004) == kvc.ERR_ALIGN
    assert call(ws_bytes=16) == kvc.ERR_WORKSPACE
    assert call(prm=kvc.default_params(flags=kvc.FLAG_SELECT_OMP)) == kvc.ERR_INVALID_ARG


def test_debug_build_compiles_and_exports():
    """The KVC_DEBUG build (kernels check data-derived indices and record
    KVC_ERR_DEBUG_BOUNDS instead of accessing out of range) compiles for
    sm_103a and exports the same interface."""
    path = kbuild.build(debug=True)
    L = ctypes.CDLL(path)
    for n in _declared():
        assert hasattr(L, n), n
    L.kvc_version.restype = ctypes.c_char_p
    assert L.kvc_version().decode().endswith("debug")
    L.kvc_status_string.argtypes = [ctypes.c_int]
    L.kvc_status_string.restype = ctypes.c_char_p
    assert b"debug" in L.kvc_status_string(kvc.ERR_DEBUG_BOUNDS)
