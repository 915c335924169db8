"""The N > 1 benchmark path on CPU: world size 2 over gloo.

Ranks run independent replicas of the workload (the path shards into
independent (sequence, KV head) units with no exchange), so the only
cross-rank steps are the barrier and the max over ranks of the step time;
the job's rate is all ranks' units over the slowest rank's time.
"""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    step_ms = [0.30, 0.42][rank]  # rank 1 is the slower one
    dist.barrier()
    worst = bench.max_over_ranks(step_ms, world)
    rate = bench.job_throughput(2_147_500_032, world, worst)
    q.put((rank, worst, rate))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_max_over_ranks_and_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, worst, rate in res:
        assert worst == pytest.approx(0.42)
        # two replicas of the long-decode bytes over the slower rank's step
        assert rate == pytest.approx(2 * 2_147_500_032 / 0.42e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.job_throughput(1e12, 1, 1000.0) == pytest.approx(1.0)
