"""Python binding of libkvc, the B300 Attention Matching KV-compaction library.

Argument marshalling only: every step of the compaction runs in the CUDA
kernels of libkvc.so (built in-tree by ``kv_cache_compaction_03_b300.build``).
PyTorch supplies device memory and streams.  There is no CPU fallback: if the
library is missing, ``lib()`` raises.

The C entry points are declared in include/kvc.h; the Python functions below
carry the same names without the ``kvc_`` prefix.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
# KVC_LIBRARY=debug loads the build whose kernels check data-derived indices
# (python -m kv_cache_compaction_03_b300.build --debug)
LIB_NAME = "libkvc_debug.so" if os.environ.get("KVC_LIBRARY") == "debug" else "libkvc.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)

# status codes (include/kvc.h)
OK = 0
ERR_INVALID_ARG = 1
ERR_ALIGN = 2
ERR_WORKSPACE = 3
ERR_CUDA = 4
ERR_NOALLOC_LIMIT = 5
NOALLOC_SCRATCH_BYTES = 64 << 20
ERR_BAD_BUDGET = 16
ERR_NOT_SPD = 17
ERR_NNLS_MAXITER = 18
ERR_NONFINITE = 19
ERR_TIMEOUT = 20
ERR_DEBUG_BOUNDS = 21

DTYPE_BF16 = 0
DTYPE_F32 = 1

WS_O, WS_LSE2, WS_SCORE, WS_W, WS_HEAD, WS_ORDER, WS_L2 = 0, 1, 2, 3, 4, 5, 6


class Problem(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("n", ctypes.c_int32), ("T", ctypes.c_int32),
                ("d", ctypes.c_int32), ("dtype", ctypes.c_int32), ("max_t", ctypes.c_int32)]


class Params(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("eps_mu", ctypes.c_float), ("eps_lambda", ctypes.c_float),
                ("nnls_max_iter", ctypes.c_int32), ("nnls_max_zero", ctypes.c_int32),
                ("refine_iters", ctypes.c_int32), ("keep_first", ctypes.c_int32),
                ("keep_last", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("wait_timeout_us", ctypes.c_uint32)]


class HeadRecord(ctypes.Structure):
    _fields_ = [("mu", ctypes.c_float), ("lam", ctypes.c_float), ("trace", ctypes.c_float),
                ("nzero", ctypes.c_int32), ("iters", ctypes.c_int32), ("pad", ctypes.c_int32 * 3)]


class KvcError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


_lib = None
EXPORTS = ("kvc_default_params", "kvc_workspace_size", "kvc_workspace_offset", "kvc_compact",
           "kvc_compact_noalloc", "kvc_compact_chunked", "kvc_workspace_size_chunked", "kvc_compact_tam",
           "kvc_workspace_size_tam", "kvc_compact_biased", "kvc_workspace_size_biased", "kvc_attend",
           "kvc_stage_times", "kvc_status_string", "kvc_version")
FLAG_STAGE_TIMING = 1
FLAG_CHOLESKY_CV = 2
FLAG_SELECT_OMP = 4


def lib() -> ctypes.CDLL:
    """Load libkvc.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_NAME} not built at {LIB_PATH}; run python -m kv_cache_compaction_03_b300.build"
                          + (" --debug" if LIB_NAME != "libkvc.so" else ""))
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    P, PP = ctypes.POINTER(Problem), ctypes.POINTER(Params)
    L.kvc_default_params.argtypes = [PP]
    L.kvc_workspace_size.argtypes = [P, PP, ctypes.POINTER(sz)]
    L.kvc_workspace_offset.argtypes = [P, PP, i32, ctypes.POINTER(sz)]
    L.kvc_compact.argtypes = [P, PP, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.kvc_compact_noalloc.argtypes = [P, PP, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.kvc_compact_chunked.argtypes = [P, PP, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.kvc_workspace_size_chunked.argtypes = [P, PP, i32, ctypes.POINTER(sz)]
    L.kvc_compact_tam.argtypes = [P, PP, vp, vp, vp, vp, i32, vp, i32, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp,
                                  vp, vp, vp, sz, vp]
    L.kvc_workspace_size_tam.argtypes = [P, PP, i32, i32, ctypes.POINTER(sz)]
    L.kvc_compact_biased.argtypes = [P, PP, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.kvc_workspace_size_biased.argtypes = [P, PP, ctypes.POINTER(sz)]
    L.kvc_attend.argtypes = [P, vp, i32, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp]
    L.kvc_stage_times.argtypes = [ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_float),
                                  ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(i32), ctypes.POINTER(i32), i32]
    L.kvc_stage_times.restype = ctypes.c_int
    L.kvc_status_string.argtypes = [ctypes.c_int]
    L.kvc_status_string.restype = ctypes.c_char_p
    L.kvc_version.restype = ctypes.c_char_p
    for f in ("kvc_default_params", "kvc_workspace_size", "kvc_workspace_offset", "kvc_compact",
              "kvc_compact_noalloc", "kvc_compact_chunked", "kvc_workspace_size_chunked", "kvc_compact_tam",
              "kvc_workspace_size_tam", "kvc_compact_biased", "kvc_workspace_size_biased", "kvc_attend"):
        getattr(L, f).restype = ctypes.c_int
    _lib = L
    return L


def status_string(code: int) -> str:
    return lib().kvc_status_string(int(code)).decode()


def version() -> str:
    return lib().kvc_version().decode()


def default_params(**kw) -> Params:
    p = Params()
    rc = lib().kvc_default_params(ctypes.byref(p))
    if rc:
        raise KvcError(rc, "kvc_default_params")
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def make_problem(H: int, n: int, T: int, d: int, dtype: int, max_t: int) -> Problem:
    return Problem(H, n, T, d, dtype, max_t)


def workspace_size(problem: Problem, params: Params | None = None) -> int:
    out = ctypes.c_size_t()
    rc = lib().kvc_workspace_size(ctypes.byref(problem), ctypes.byref(params) if params else None, ctypes.byref(out))
    if rc:
        raise KvcError(rc, "kvc_workspace_size")
    return out.value


def workspace_size_chunked(problem: Problem, params: Params | None, chunks: int) -> int:
    out = ctypes.c_size_t()
    rc = lib().kvc_workspace_size_chunked(ctypes.byref(problem), ctypes.byref(params) if params else None,
                                          int(chunks), ctypes.byref(out))
    if rc:
        raise KvcError(rc, "kvc_workspace_size_chunked")
    return out.value


def workspace_offset(problem: Problem, params: Params | None, item: int) -> int:
    out = ctypes.c_size_t()
    rc = lib().kvc_workspace_offset(ctypes.byref(problem), ctypes.byref(params) if params else None, item,
                                    ctypes.byref(out))
    if rc:
        raise KvcError(rc, "kvc_workspace_offset")
    return out.value


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def compact(problem: Problem, params: Params | None, Q_ref, K, V, budgets, offsets, idx_out, C_k, beta, C_v,
            head_status, workspace, workspace_bytes: int, stream=None) -> int:
    """kvc_compact on caller-owned buffers (torch tensors or raw device pointers).
    Returns the call-level status (0 = enqueued)."""
    return lib().kvc_compact(ctypes.byref(problem), ctypes.byref(params) if params else None,
                             _ptr(Q_ref), _ptr(K), _ptr(V), _ptr(budgets), _ptr(offsets), _ptr(idx_out),
                             _ptr(C_k), _ptr(beta), _ptr(C_v), _ptr(head_status), _ptr(workspace),
                             int(workspace_bytes), _stream(stream))


def compact_noalloc(problem: Problem, params: Params | None, Q_ref, K, V, budgets, offsets, idx_out, C_k, beta,
                    C_v, head_status, stream=None) -> int:
    """kvc_compact_noalloc: kvc_compact with the library's fixed device scratch
    (no workspace argument; for callers that cannot allocate device memory).
    Returns the call-level status (0 = enqueued)."""
    return lib().kvc_compact_noalloc(ctypes.byref(problem), ctypes.byref(params) if params else None,
                                     _ptr(Q_ref), _ptr(K), _ptr(V), _ptr(budgets), _ptr(offsets), _ptr(idx_out),
                                     _ptr(C_k), _ptr(beta), _ptr(C_v), _ptr(head_status), _stream(stream))


def compact_chunked(problem: Problem, params: Params | None, chunks: int, Q_ref, K, V, budgets, offsets, idx_out,
                    C_k, beta, C_v, head_status, workspace, workspace_bytes: int, stream=None) -> int:
    """kvc_compact_chunked: every head's cache cut into `chunks` contiguous
    chunks, each compacted against the head's reference queries.  Returns the
    call-level status (0 = enqueued)."""
    return lib().kvc_compact_chunked(ctypes.byref(problem), ctypes.byref(params) if params else None, int(chunks),
                                     _ptr(Q_ref), _ptr(K), _ptr(V), _ptr(budgets), _ptr(offsets), _ptr(idx_out),
                                     _ptr(C_k), _ptr(beta), _ptr(C_v), _ptr(head_status), _ptr(workspace),
                                     int(workspace_bytes), _stream(stream))


def workspace_size_tam(problem: Problem, params: Params | None, n_win: int, nseg: int) -> int:
    out = ctypes.c_size_t()
    rc = lib().kvc_workspace_size_tam(ctypes.byref(problem), ctypes.byref(params) if params else None, int(n_win),
                                      int(nseg), ctypes.byref(out))
    if rc:
        raise KvcError(rc, "kvc_workspace_size_tam")
    return out.value


def compact_tam(problem: Problem, params: Params | None, Q_ref, K, V, Q_win, n_win: int, seg_bounds, nseg: int,
                pivot_c: float, budgets, offsets, idx_out, C_k, beta, C_v, head_status, seg_budgets_out, pivots_out,
                workspace, workspace_bytes: int, stream=None) -> int:
    """kvc_compact_tam: thought-aware budgets per segment and exact pivots.
    Returns the call-level status (0 = enqueued)."""
    return lib().kvc_compact_tam(ctypes.byref(problem), ctypes.byref(params) if params else None, _ptr(Q_ref),
                                 _ptr(K), _ptr(V), _ptr(Q_win), int(n_win), _ptr(seg_bounds), int(nseg),
                                 float(pivot_c), _ptr(budgets), _ptr(offsets), _ptr(idx_out), _ptr(C_k), _ptr(beta),
                                 _ptr(C_v), _ptr(head_status), _ptr(seg_budgets_out), _ptr(pivots_out),
                                 _ptr(workspace), int(workspace_bytes), _stream(stream))


def workspace_size_biased(problem: Problem, params: Params | None = None) -> int:
    out = ctypes.c_size_t()
    rc = lib().kvc_workspace_size_biased(ctypes.byref(problem), ctypes.byref(params) if params else None,
                                         ctypes.byref(out))
    if rc:
        raise KvcError(rc, "kvc_workspace_size_biased")
    return out.value


def compact_biased(problem: Problem, params: Params | None, Q_ref, K, bias, V, budgets, offsets, idx_out, C_k, beta,
                   C_v, head_status, workspace, workspace_bytes: int, stream=None) -> int:
    """kvc_compact_biased: compaction of a cache whose keys carry biases and
    whose values are fp32 (periodic compaction).  Returns the call-level
    status (0 = enqueued)."""
    return lib().kvc_compact_biased(ctypes.byref(problem), ctypes.byref(params) if params else None, _ptr(Q_ref),
                                    _ptr(K), _ptr(bias), _ptr(V), _ptr(budgets), _ptr(offsets), _ptr(idx_out),
                                    _ptr(C_k), _ptr(beta), _ptr(C_v), _ptr(head_status), _ptr(workspace),
                                    int(workspace_bytes), _stream(stream))


def attend(problem: Problem, Q, n_q: int, C_k, beta, C_v, offsets, O_out, head_status, scale: float = 0.0,
           stream=None) -> int:
    """kvc_attend on caller-owned buffers.  Returns the call-level status."""
    return lib().kvc_attend(ctypes.byref(problem), _ptr(Q), int(n_q), _ptr(C_k), _ptr(beta), _ptr(C_v),
                            _ptr(offsets), _ptr(O_out), _ptr(head_status), float(scale), _stream(stream))


def stage_times(cap: int = 32):
    """[(name, ms, kernel_launches)] of the last timed kvc_compact on this thread,
    and the launch count of the last kvc_compact call."""
    n = ctypes.c_int32()
    ms = (ctypes.c_float * cap)()
    names = (ctypes.c_char_p * cap)()
    counts = (ctypes.c_int32 * cap)()
    launches = ctypes.c_int32()
    rc = lib().kvc_stage_times(ctypes.byref(n), ms, names, counts, ctypes.byref(launches), cap)
    if rc:
        raise KvcError(rc, "kvc_stage_times")
    return [(names[i].decode(), float(ms[i]), int(counts[i])) for i in range(min(n.value, cap))], launches.value


# ------------------------------------------------------------------ helpers
@dataclass
class Compacted:
    """Outputs of one kvc_compact or kvc_compact_chunked call (device
    tensors).  For a chunked call, offsets / head_status are per chunk,
    `problem` is the per-chunk problem (its workspace layout) and head h's
    merged cache is rows [offsets[h*chunks], offsets[(h+1)*chunks])."""
    idx: object
    C_k: object
    beta: object
    C_v: object
    offsets: object
    head_status: object
    workspace: object
    problem: Problem
    params: Params
    chunks: int = 1

    def head_offsets(self):
        """int32 [H+1]: each head's row range in the (merged) compact cache."""
        return self.offsets if self.chunks == 1 else self.offsets[::self.chunks].contiguous()


def torch_dtype_code(dt) -> int:
    import torch
    if dt == torch.bfloat16:
        return DTYPE_BF16
    if dt == torch.float32:
        return DTYPE_F32
    raise ValueError(f"unsupported dtype {dt}")


def compact_tensors(Q_ref, K, V, budgets, params: Params | None = None, stream=None) -> Compacted:
    """Allocate outputs and workspace with torch, then call kvc_compact.

    Q_ref [H][n][d], K/V [H][T][d] (bf16 or fp32, contiguous, on the same CUDA
    device); budgets int32 [H] on the device.  Work is enqueued on `stream`.
    """
    import torch
    H, n, d = Q_ref.shape
    T = K.shape[1]
    dev = Q_ref.device
    b64 = budgets.to(torch.int64)
    offsets = torch.zeros(H + 1, dtype=torch.int32, device=dev)
    offsets[1:] = torch.cumsum(b64, 0).to(torch.int32)
    total = int(offsets[-1].item())
    max_t = int(b64.max().item())
    prob = make_problem(H, n, T, d, torch_dtype_code(Q_ref.dtype), max_t)
    prm = params if params is not None else default_params()
    ws_bytes = workspace_size(prob, prm)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    idx = torch.empty(total, dtype=torch.int32, device=dev)
    Ck = torch.empty(total, d, dtype=Q_ref.dtype, device=dev)
    beta = torch.empty(total, dtype=torch.float32, device=dev)
    Cv = torch.empty(total, d, dtype=torch.float32, device=dev)
    status = torch.empty(H, dtype=torch.int32, device=dev)
    rc = compact(prob, prm, Q_ref, K, V, budgets, offsets, idx, Ck, beta, Cv, status, ws, ws_bytes, stream)
    if rc:
        raise KvcError(rc, "kvc_compact")
    return Compacted(idx, Ck, beta, Cv, offsets, status, ws, prob, prm)


def compact_biased_tensors(Q_ref, K, bias, V, budgets, params: Params | None = None, stream=None) -> Compacted:
    """Allocate outputs and workspace with torch, then call kvc_compact_biased.

    Q_ref [H][n][d] and K [H][T][d] (bf16 or fp32), bias fp32 [H][T], V fp32
    [H][T][d], budgets int32 [H], all on the same CUDA device.
    """
    import torch
    H, n, d = Q_ref.shape
    T = K.shape[1]
    dev = Q_ref.device
    b64 = budgets.to(torch.int64)
    offsets = torch.zeros(H + 1, dtype=torch.int32, device=dev)
    offsets[1:] = torch.cumsum(b64, 0).to(torch.int32)
    total = int(offsets[-1].item())
    max_t = int(b64.max().item())
    prob = make_problem(H, n, T, d, torch_dtype_code(Q_ref.dtype), max_t)
    prm = params if params is not None else default_params()
    ws_bytes = workspace_size_biased(prob, prm)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    idx = torch.empty(total, dtype=torch.int32, device=dev)
    Ck = torch.empty(total, d, dtype=Q_ref.dtype, device=dev)
    beta = torch.empty(total, dtype=torch.float32, device=dev)
    Cv = torch.empty(total, d, dtype=torch.float32, device=dev)
    status = torch.empty(H, dtype=torch.int32, device=dev)
    rc = compact_biased(prob, prm, Q_ref, K, bias, V, budgets, offsets, idx, Ck, beta, Cv, status, ws, ws_bytes,
                        stream)
    if rc:
        raise KvcError(rc, "kvc_compact_biased")
    return Compacted(idx, Ck, beta, Cv, offsets, status, ws, prob, prm)


def compact_chunked_tensors(Q_ref, K, V, budgets, params: Params | None = None, stream=None) -> Compacted:
    """Allocate outputs and workspace with torch, then call kvc_compact_chunked.

    Q_ref [H][n][d], K/V [H][T][d]; budgets int32 [H][chunks] on the device
    (the chunk count is its second dimension; T must be a multiple of it).
    """
    import torch
    H, n, d = Q_ref.shape
    T = K.shape[1]
    C = budgets.shape[1]
    dev = Q_ref.device
    flat = budgets.reshape(-1).contiguous()
    b64 = flat.to(torch.int64)
    offsets = torch.zeros(H * C + 1, dtype=torch.int32, device=dev)
    offsets[1:] = torch.cumsum(b64, 0).to(torch.int32)
    total = int(offsets[-1].item())
    max_t = int(b64.max().item())
    prob = make_problem(H, n, T, d, torch_dtype_code(Q_ref.dtype), max_t)
    prm = params if params is not None else default_params()
    ws_bytes = workspace_size_chunked(prob, prm, C)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    idx = torch.empty(total, dtype=torch.int32, device=dev)
    Ck = torch.empty(total, d, dtype=Q_ref.dtype, device=dev)
    beta = torch.empty(total, dtype=torch.float32, device=dev)
    Cv = torch.empty(total, d, dtype=torch.float32, device=dev)
    status = torch.empty(H * C, dtype=torch.int32, device=dev)
    rc = compact_chunked(prob, prm, C, Q_ref, K, V, flat, offsets, idx, Ck, beta, Cv, status, ws, ws_bytes, stream)
    if rc:
        raise KvcError(rc, "kvc_compact_chunked")
    chunk_prob = make_problem(H * C, n, T // C, d, prob.dtype, max_t)
    return Compacted(idx, Ck, beta, Cv, offsets, status, ws, chunk_prob, prm, C)


def compact_tam_tensors(Q_ref, K, V, Q_win, seg_bounds, budgets, pivot_c: float, params: Params | None = None,
                        stream=None):
    """Allocate outputs and workspace with torch, then call kvc_compact_tam.
    seg_bounds: int32 [nseg + 1] on the device.  Returns (Compacted,
    seg_budgets [H][nseg] int32, pivots [H][T] uint8)."""
    import torch
    H, n, d = Q_ref.shape
    T = K.shape[1]
    nw = Q_win.shape[1]
    nseg = seg_bounds.shape[0] - 1
    dev = Q_ref.device
    b64 = budgets.to(torch.int64)
    offsets = torch.zeros(H + 1, dtype=torch.int32, device=dev)
    offsets[1:] = torch.cumsum(b64, 0).to(torch.int32)
    total = int(offsets[-1].item())
    max_t = int(b64.max().item())
    prob = make_problem(H, n, T, d, torch_dtype_code(Q_ref.dtype), max_t)
    prm = params if params is not None else default_params()
    ws_bytes = workspace_size_tam(prob, prm, nw, nseg)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    idx = torch.empty(total, dtype=torch.int32, device=dev)
    Ck = torch.empty(total, d, dtype=Q_ref.dtype, device=dev)
    beta = torch.empty(total, dtype=torch.float32, device=dev)
    Cv = torch.empty(total, d, dtype=torch.float32, device=dev)
    status = torch.empty(H, dtype=torch.int32, device=dev)
    segb = torch.empty(H, nseg, dtype=torch.int32, device=dev)
    piv = torch.empty(H, T, dtype=torch.uint8, device=dev)
    rc = compact_tam(prob, prm, Q_ref, K, V, Q_win, nw, seg_bounds, nseg, pivot_c, budgets, offsets, idx, Ck, beta,
                     Cv, status, segb, piv, ws, ws_bytes, stream)
    if rc:
        raise KvcError(rc, "kvc_compact_tam")
    return Compacted(idx, Ck, beta, Cv, offsets, status, ws, prob, prm), segb, piv


def workspace_view(c: Compacted, item: int, count: int, dtype):
    """A typed view of an intermediate inside a finished call's workspace."""
    import torch
    off = workspace_offset(c.problem, c.params, item)
    esz = torch.empty((), dtype=dtype).element_size()
    return c.workspace[off: off + count * esz].view(dtype)


def attend_tensors(Q, c: Compacted, scale: float = 0.0, stream=None):
    """softmax(Q C_k^T * scale + beta) C_v per head (over the merged cache of a
    chunked call); returns (O [H][n_q][d] fp32, status)."""
    import torch
    H, nq, d = Q.shape
    O = torch.empty(H, nq, d, dtype=torch.float32, device=Q.device)
    st = torch.empty(H, dtype=torch.int32, device=Q.device)
    prob = make_problem(H, nq, 1, d, torch_dtype_code(Q.dtype), 1)
    rc = attend(prob, Q, nq, c.C_k, c.beta, c.C_v, c.head_offsets(), O, st, scale, stream)
    if rc:
        raise KvcError(rc, "kvc_attend")
    return O, st
