"""The multi-GPU mode's host logic on CPU: two gloo ranks.

The path shards by solve with no exchange step (replicas), so what N > 1
adds is host code: each rank's slice of the problem stream, the max-over-
ranks timing reduction and the whole-job throughput.  Two spawned processes
run it over gloo on 127.0.0.1."""
import multiprocessing as mp
import socket

import numpy as np
import pytest

from trajectory_optimization_kkt_gb300.replicas import Replica, job_throughput, max_over_ranks
from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch

BATCH = 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        r = Replica(world, rank, rank)
        w = WORKLOADS[1]
        mine = make_batch(w, M=BATCH, first_solve=r.first_solve(BATCH))
        # per-rank "times": the job takes the slowest
        local = [10.0 + 5.0 * rank, 3.0 - rank]
        slowest = max_over_ranks(local, dist)
        out.put((rank, list(r.solves(BATCH)), mine["Q"].tobytes(), slowest,
                 job_throughput(BATCH, world, slowest[0])))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_the_stream_and_reduce_the_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, q0, t0, v0), (r1, s1, q1, t1, v1) = res
    assert (r0, r1) == (0, 1)
    # disjoint, contiguous slices of one problem stream
    assert s0 == [0, 1, 2] and s1 == [3, 4, 5]
    whole = make_batch(WORKLOADS[1], M=2 * BATCH)
    shape = whole["Q"].shape[1:]
    np.testing.assert_array_equal(np.frombuffer(q0, np.float32).reshape((BATCH,) + shape),
                                  whole["Q"][:BATCH])
    np.testing.assert_array_equal(np.frombuffer(q1, np.float32).reshape((BATCH,) + shape),
                                  whole["Q"][BATCH:])
    # both ranks see the slowest rank's time, element by element
    assert t0 == t1 == [15.0, 3.0]
    # all ranks' solves over the slowest time
    assert v0 == v1 == pytest.approx(2 * BATCH / 0.015)


def test_single_rank_needs_no_process_group():
    r = Replica(1, 0, 0)
    assert list(r.solves(4)) == [0, 1, 2, 3]
    assert max_over_ranks([2.5, 1.0]) == [2.5, 1.0]
    assert job_throughput(256, 1, 4.0) == pytest.approx(64000.0)
