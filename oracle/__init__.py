"""Float64 CPU oracle for Attention Matching KV-cache compaction.

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and by
the CPU-baseline / reference legs of bench.py.  The GPU library never imports,
links or runs anything here, and this package shares no code with it.

Every function is pinned by tests in tests/test_oracle_pins.py against facts
that do not come from the oracle itself (brute force on tiny inputs, closed
forms, KKT conditions, library solvers on special cases, and the page's own
q = 0 example).  The end-to-end quality of a compaction with t < T (how close
the compacted outputs are to the full ones) has no printed value on the pages:
that quantity is reported, not asserted (parity unpinned).
"""
from .am import (  # noqa: F401
    EPS_LAMBDA_DEFAULT, EPS_MU_DEFAULT, HeadResult, attend, attend_full,
    attention_reference, biased_softmax, compact_head, decode, fit_beta,
    fit_values, key_scores, mass_matrix, nnls_bpp, nnls_kkt_violation,
    select_top_t,
)
from .chunked import compact_chunked  # noqa: F401
from .omp import compact_head_omp, omp_residual, omp_select  # noqa: F401
from .periodic import attention_biased, compact_head_biased, periodic_compaction  # noqa: F401
from .tam import compact_head_tam, plan_head  # noqa: F401
