"""bench.py's multi-rank bookkeeping, on the host: two gloo ranks agree on the slowest rank's time
and the job rate counts every rank's units (one process per GPU runs independent replicas)."""
import os
import socket

import torch


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
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"))
    q.put((rank, ms, bench.job_rate(3840, world, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(12.5, torch.device("cpu")) == 12.5
    assert bench.job_rate(3840, 1, 50.0) == 3840 / 0.05


def test_two_ranks_max_and_job_rate():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    assert [r[1] for r in res] == [15.0, 15.0]           # both ranks report the slower rank's time
    assert all(abs(r[2] - 2 * 3840 / 0.015) < 1e-6 for r in res)
