"""The five synthetic workloads the compaction path is tested and measured on.

Each workload is a batch of independent KV heads.  A head is addressed by
(sequence, layer, kv_head); its inputs are drawn from a seed derived from
that address, so any single head can be regenerated on its own.

The shapes follow the long-context settings that the Attention Matching
explainer ("Fast KV Compaction via Attention Matching", gist.science,
sections 2 and 4) talks about: Llama-3-8B-like layers (8 KV heads, GQA 4,
d=128), long caches, 10x-50x compaction, non-uniform per-head budgets, and a
reasoning-trace cache built from segments (the segment structure follows the
"Thought-Aware KV Cache Compaction" explainer, section 2A).
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    cfg_id: int
    name: str
    seqs: int             # independent sequences
    layers: int           # layers per sequence
    kv_heads: int         # KV heads per layer
    n: int                # reference queries per KV head (GQA group stacked)
    T: int                # cached tokens per head
    d: int                # head dim
    t: int | None         # uniform budget (None: non-uniform budgets)
    dtype: str            # "f32" or "bf16"
    gqa: int = 1          # query heads per KV head (rows are stacked in n)
    rank: int = 16        # rank of the low-rank part of K (uniform)
    rank_by_layer: tuple[int, int] | None = None   # (lo, hi): rank varies linearly over layers
    scale_range: tuple[float, float] | None = None  # per-head K scale ~ U(lo, hi)
    sinks: int = 0        # leading tokens whose K rows are scaled x4
    rope_theta: float | None = None
    segments: int = 0     # >0: K built from this many segments, each its own basis
    seg_rank: int = 0
    keep_first: int = 0   # forced keeps (always in the compacted set)
    keep_last: int = 0
    budget_frac: float = 0.0   # non-uniform budgets: mean budget = budget_frac * T
    budget_floor: int = 0      # floor on the non-forced part of a budget
    n_test: int = 256          # held-out queries per head
    noise_k: float = 0.3       # K = G U + noise_k * N(0,1)
    q_noise_var: float = 0.5   # Q = K[j] + N(0, q_noise_var)
    seq_offset: int = 0        # first sequence index (replicas draw distinct sequences)

    @property
    def H(self) -> int:
        return self.seqs * self.layers * self.kv_heads

    def head_address(self, h: int) -> tuple[int, int, int]:
        """(sequence, layer, kv_head) of flat head index h."""
        per_seq = self.layers * self.kv_heads
        s, r = divmod(h, per_seq)
        layer, kv = divmod(r, self.kv_heads)
        return s + self.seq_offset, layer, kv


WORKLOADS: dict[int, Workload] = {
    1: Workload(cfg_id=1, name="tiny-1head-T1024-d64-fp32", seqs=1, layers=1, kv_heads=1,
                n=256, T=1024, d=64, t=64, dtype="f32", rank=16, sinks=4),
    2: Workload(cfg_id=2, name="llama3-8b-layer-T8192", seqs=1, layers=1, kv_heads=8,
                n=4096, T=8192, d=128, t=820, dtype="bf16", gqa=4, rank=32, sinks=4,
                rope_theta=500000.0),
    3: Workload(cfg_id=3, name="llama3-8b-32layer-cache-T32768", seqs=1, layers=32, kv_heads=8,
                n=8192, T=32768, d=128, t=655, dtype="bf16", gqa=4,
                rank_by_layer=(16, 64), scale_range=(0.5, 2.0), sinks=4,
                rope_theta=500000.0),
    4: Workload(cfg_id=4, name="reasoning-trace-T16384-nonuniform", seqs=1, layers=28, kv_heads=4,
                n=2048, T=16384, d=128, t=None, dtype="bf16", segments=64, seg_rank=8,
                keep_first=4, keep_last=64, budget_frac=0.1, budget_floor=32),
    5: Workload(cfg_id=5, name="serving-batch-16x8-T4096", seqs=16, layers=1, kv_heads=8,
                n=1024, T=4096, d=128, t=1024, dtype="bf16", gqa=4, rank=32, sinks=4,
                rope_theta=500000.0),
}


def small_variant(w: Workload, *, H: int | None = None, n: int | None = None,
                  T: int | None = None, t: int | None = None, d: int | None = None,
                  dtype: str | None = None) -> Workload:
    """A reduced copy of a workload (same generator recipe, smaller shapes).

    Used by tests that need many tiles and a ragged tail but must finish in
    seconds on the CPU.  H counts heads of one sequence and one layer.
    """
    from dataclasses import replace
    kw = {}
    if H is not None:
        kw.update(seqs=1, layers=1, kv_heads=H)
    if n is not None:
        kw["n"] = n
    if T is not None:
        kw["T"] = T
    if t is not None:
        kw["t"] = t
    if d is not None:
        kw["d"] = d
    if dtype is not None:
        kw["dtype"] = dtype
    if w.segments and T is not None:
        kw["segments"] = max(1, min(w.segments, T // 64))
    return replace(w, name=w.name + "-small", **kw)
