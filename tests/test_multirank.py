"""The N > 1 path of bench.py on the CPU: two gloo ranks.

Heads are independent problems, so N GPUs run N replicas that compact
disjoint sequences with no exchange on the data path; the only cross-rank
traffic is the timing barrier and the max-reduction of the step time.  These
tests run that host logic with world_size 2 over gloo (no GPU).
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from workloads import WORKLOADS, small_variant
from workloads.gen import head_inputs


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        base = small_variant(WORKLOADS[5], H=2, n=16, T=32, t=8)
        w = bench.rank_workload(base, rank, world)
        addrs = [w.head_address(h) for h in range(w.H)]
        first = head_inputs(w, 0, with_test=False)["K"]
        # each rank reports a different step time; every rank must see the max
        t = bench.max_over_ranks(10.0 + rank, dist, torch.device("cpu"))
        dist.barrier()
        out[rank] = (addrs, first.tobytes(), t)
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        codes = [p.exitcode for p in procs]
        res = dict(out)
    assert codes == [0, 0], codes
    return res


def test_ranks_compact_disjoint_sequences(two_ranks):
    a0, k0, _ = two_ranks[0]
    a1, k1, _ = two_ranks[1]
    assert set(a0).isdisjoint(set(a1))
    assert {s for s, _, _ in a0} == {0} and {s for s, _, _ in a1} == {1}
    assert k0 != k1                      # distinct seeds give distinct caches


def test_step_time_is_max_over_ranks(two_ranks):
    assert two_ranks[0][2] == 11.0 and two_ranks[1][2] == 11.0


def test_single_rank_is_the_base_workload():
    base = WORKLOADS[2]
    assert bench.rank_workload(base, 0, 1) is base
    assert bench.max_over_ranks(3.5, None, None) == 3.5


def test_replica_of_rank_r_equals_base_sequence_r():
    """Rank r's heads are exactly the base generator's sequence r (weak
    scaling reproduces a larger batch of the same workload)."""
    base = small_variant(WORKLOADS[5], H=2, n=16, T=32, t=8)
    w1 = bench.rank_workload(base, 1, 2)
    from dataclasses import replace
    big = replace(base, seqs=2)
    x = head_inputs(w1, 0, with_test=False)["K"]
    y = head_inputs(big, base.H, with_test=False)["K"]    # first head of sequence 1
    np.testing.assert_array_equal(x, y)
