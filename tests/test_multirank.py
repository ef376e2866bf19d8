"""Multi-rank (replica) host logic of bench.py on CPU: world size 2, gloo backend.

Each rank runs its own replica of the workload; the job time is the largest rank time and
the job throughput counts every rank's work.  No GPU and no data-path collective involved.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = [120.0, 150.0][rank]
    job_ms = bench.max_over_ranks(local_ms, world, device="cpu")
    tput = bench.job_throughput(10 ** 12, 4, world, job_ms)
    q.put((rank, job_ms, tput))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_time_is_max_and_work_is_summed():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, job_ms, tput in res:
        assert job_ms == 150.0
        # 2 ranks x 4 steps x 1e12 flop in 0.150 s
        assert tput == pytest.approx(2 * 4 * 1e12 / 0.150 / 1e12)


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_throughput(2 * 10 ** 12, 3, 1, 1000.0) == pytest.approx(6.0)
