"""Whole-call input generation: every head of a workload, stacked.

Heads are independent draws (see gen.py), so they are generated in parallel
worker processes (spawn start method) that write straight into shared memory.
"""
from __future__ import annotations

import os
from concurrent.futures import ProcessPoolExecutor
from multiprocessing import get_context, shared_memory

import numpy as np

from .configs import WORKLOADS, Workload
from .gen import head_inputs

_FIELDS = ("Q", "K", "V", "Qt")


def _shapes(w: Workload) -> dict:
    H = w.H
    return {"Q": (H, w.n, w.d), "K": (H, w.T, w.d), "V": (H, w.T, w.d), "Qt": (H, w.n_test, w.d)}


def _np_dtype(w: Workload):
    return np.uint16 if w.dtype == "bf16" else np.float32


def _work(args):
    cfg_id, overrides, heads, shm_names = args
    w = _rebuild(cfg_id, overrides)
    dt = _np_dtype(w)
    shapes = _shapes(w)
    bufs = {k: shared_memory.SharedMemory(name=shm_names[k]) for k in _FIELDS}
    try:
        arrs = {k: np.ndarray(shapes[k], dtype=dt, buffer=bufs[k].buf) for k in _FIELDS}
        for h in heads:
            x = head_inputs(w, h)
            for k in _FIELDS:
                arrs[k][h] = x[k]
    finally:
        for b in bufs.values():
            b.close()
    return len(heads)


def _rebuild(cfg_id, overrides):
    from dataclasses import replace
    w = WORKLOADS[cfg_id]
    return replace(w, **overrides) if overrides else w


def generate(w: Workload, workers: int | None = None) -> dict:
    """All heads of w: dict of stacked arrays Q [H][n][d], K/V [H][T][d], Qt [H][n_test][d]."""
    from dataclasses import asdict
    base = WORKLOADS[w.cfg_id]
    overrides = {k: v for k, v in asdict(w).items() if getattr(base, k) != v}
    dt = _np_dtype(w)
    shapes = _shapes(w)
    H = w.H
    if workers is None:
        workers = min(H, max(1, (os.cpu_count() or 1)))
    if workers <= 1 or H <= 2:
        out = {k: np.empty(shapes[k], dtype=dt) for k in _FIELDS}
        for h in range(H):
            x = head_inputs(w, h)
            for k in _FIELDS:
                out[k][h] = x[k]
        return out
    itemsize = np.dtype(dt).itemsize
    shms = {k: shared_memory.SharedMemory(create=True, size=int(np.prod(shapes[k])) * itemsize) for k in _FIELDS}
    try:
        names = {k: s.name for k, s in shms.items()}
        chunks = [list(range(i, H, workers)) for i in range(workers)]
        with ProcessPoolExecutor(max_workers=workers, mp_context=get_context("spawn")) as ex:
            done = sum(ex.map(_work, [(w.cfg_id, overrides, c, names) for c in chunks if c]))
        assert done == H
        out = {k: np.ndarray(shapes[k], dtype=dt, buffer=shms[k].buf).copy() for k in _FIELDS}
    finally:
        for s in shms.values():
            s.close()
            s.unlink()
    return out
