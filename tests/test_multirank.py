"""The N > 1 benchmark path on CPU: two gloo ranks run independent replicas; the job time is the
slowest rank's, the job throughput counts every rank's work, and only rank 0 reports."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [1.0 + rank, 10.0 - rank]                 # each rank's own timings
    got = bench.reduce_max(ms, dist, torch.device("cpu"))
    tput = bench.job_throughput(1e12, world, got[0])
    q.put((rank, got, tput))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_max_time_and_job_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, tput in res:
        assert got == [2.0, 10.0]                  # max over ranks, element-wise
        assert abs(tput - 1e12 * 2 / 2e-3 / 1e12) < 1e-9


def test_reference_arm_rank_nonzero_does_no_work(capsys):
    import bench

    class A:
        steps, warmup, gpus = 1, 0, 2
    bench.run_reference(A, rank=1)
    assert capsys.readouterr().out == ""
