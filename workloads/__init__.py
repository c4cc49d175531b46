"""Seeded synthetic workloads shared by the oracle tests and the GPU path."""
from .configs import WORKLOADS, Workload, small_variant  # noqa: F401
from .gen import budgets, compacted_cache_extras, forced_mask, head_inputs, segment_bounds, window_queries  # noqa: F401
