"""Multi-rank host logic of bench.py on CPU: world_size-2 gloo process groups.

The bench runs one independent replica of the forward per GPU (the path does
not shard: no data-path collective); its only collectives are the max over
ranks of the timed region and a barrier.  These tests run that logic on two
CPU processes with the gloo backend."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each replica timed K steps in a different time; the job took the slowest one's
        local_ms = 100.0 + 25.0 * rank
        got = bench.max_over_ranks(local_ms)
        rate = bench.whole_job_rate(2048 * 10, world, got)
        dist.barrier()
        q.put((rank, got, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, got, rate in res:
        assert got == 125.0                       # max over ranks, seen identically by every rank
        assert rate == pytest.approx(2 * 2048 * 10 / 0.125)   # all ranks' tokens / slowest time


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5       # no process group: the local value
    assert bench.whole_job_rate(1000, 1, 500.0) == pytest.approx(2000.0)


def _ref_rank1(q):
    os.environ.update(RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    sys.path.insert(0, ROOT)
    import bench
    from moe_expert_ffn_route_gb300 import synth

    class Args:
        steps, warmup = 1, 1
    bench.run_reference(Args, synth.WORKLOADS["tiny"])   # returns at once: only rank 0 runs the oracle
    q.put("done")


def test_reference_arm_runs_on_rank0_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_ref_rank1, args=(q,))
    p.start()
    p.join(timeout=60)
    assert p.exitcode == 0 and q.get(timeout=5) == "done"
