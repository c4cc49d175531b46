"""A compaction through the debug build (libkvc_debug.so, compiled with
KVC_DEBUG: kernels check the indices they read from data against the
buffers those index and record KVC_ERR_DEBUG_BOUNDS instead of an
out-of-range access).  On valid inputs no check may fire and the results
must meet the usual parity tolerances.  Runs in a child process, because
the binding loads one library per process (KVC_LIBRARY=debug)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
sys.path.insert(0, "tests")
import numpy as np
import kv_cache_compaction_03_b300 as kvc
from parity import compare_head, head_queries, run_gpu, run_oracle_head
from workloads import WORKLOADS, small_variant
from workloads.batch import generate
assert kvc.version().endswith("debug"), kvc.version()
for w in (small_variant(WORKLOADS[2], H=3, n=320, T=1000, t=100),
          small_variant(WORKLOADS[4], H=2, n=256, T=1024),
          small_variant(WORKLOADS[1], H=2, n=128, T=500, t=40)):
    x = generate(w, workers=1)
    g, _ = run_gpu(w, inputs=x)
    assert np.all(g["status"] == 0), g["status"]
    from workloads import budgets
    b = budgets(w)
    for h in range(w.H):
        r, Ohat = run_oracle_head(w, x, h, int(b[h]))
        compare_head(g, h, r, Ohat, {"head": h}, Q=head_queries(w, x, h))
print("debug build ok")
"""


def test_debug_build_compaction():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_compaction_03_b300 import build
    build.build(debug=True)
    env = dict(os.environ, KVC_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "debug build ok" in r.stdout
