"""Rules on the CUDA sources that no compiler checks (no GPU needed).

* Every kernel launched with programmatic dependent launch (`launch_dep`,
  or the launch attribute in a hand-built configuration) must call
  `grid_dependency_wait()` before it touches memory: such a launch may start
  while the previous kernel is still draining, and only that wait orders it
  after the previous kernel's writes.
* No source calls the batched memory-copy entry points of the CUDA runtime or
  driver (they are not used anywhere in this library; copies are one
  `cudaMemcpyAsync` each, or a gather kernel)."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "kv_cache_compaction_03_b300", "csrc")


def _sources():
    out = {}
    for p in sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))):
        with open(p) as fh:
            out[os.path.basename(p)] = fh.read()
    return out


def _kernel_body_head(src, name, lines=6):
    """The first `lines` statements of kernel `name`'s body (None if absent)."""
    m = re.search(r"__global__[^;{]*?\b" + re.escape(name) + r"\s*\(", src)
    if m is None:
        return None
    brace = src.index("{", m.end())
    return "\n".join(src[brace + 1:].split("\n")[: lines + 1])


def test_dependent_launches_wait_for_their_predecessor():
    srcs = _sources()
    every = "\n".join(srcs.values())
    launched = set()
    for src in srcs.values():
        for m in re.finditer(r"launch_dep\(\s*([A-Za-z_][A-Za-z_0-9]*)", src):
            if m.group(1) != "void":            # the helper's own declaration
                launched.add(m.group(1))
    # `kern` is a local alias for the key-score kernel template
    assert "kern" in launched
    launched.discard("kern")
    launched.add("k_colscore_tc")
    # the matching-pursuit step is launched with the attribute in its own
    # cluster configuration
    assert "cudaLaunchAttributeProgrammaticStreamSerialization" in srcs["omp.cu"]
    launched.add("k_omp_step")
    assert len(launched) >= 20, sorted(launched)
    missing = []
    for name in sorted(launched):
        head = _kernel_body_head(every, name, lines=8)
        assert head is not None, f"kernel {name} not found"
        if "grid_dependency_wait();" not in head:
            missing.append(name)
    assert not missing, f"launched dependent without a wait at the top: {missing}"


def test_no_batched_copy_entry_points():
    names = [p + "BatchAsync" for p in ("cudaMemcpy", "cudaMemcpy3D", "cuMemcpy", "cuMemcpy3D")]
    for fname, src in _sources().items():
        for nm in names:
            assert nm not in src, f"{fname} names {nm}"
