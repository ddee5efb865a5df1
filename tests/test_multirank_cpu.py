"""The N>1 host logic of bench.py on CPU: two gloo ranks each time their own
replica; the job reports the slowest rank's step time and the whole-job
throughput; the reference arm prints from rank 0 only."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [2.5, 4.0][rank]
    ms = bench.max_over_ranks(local_ms, dist, "cpu")
    v = bench.job_value(ms, world, 32)
    q.put((rank, ms, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_slowest_rank_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, v in got:
        assert ms == 4.0
        assert v == pytest.approx(2 * 32 / 4.0e-3)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.0, None) == 3.0
    assert bench.job_value(2.0, 1, 32) == pytest.approx(16000.0)
