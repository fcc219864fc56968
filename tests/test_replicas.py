"""Multi-GPU runs are replicas (one model copy per rank, no data-path
collective); the only cross-rank step is the timing aggregate, checked here
with two gloo ranks on the CPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r ran for 100 (r + 1) ms and produced 50 tokens
    q.put((rank, bench.job_rate(100.0 * (rank + 1), 50, world)))
    dist.destroy_process_group()


def test_job_rate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        rate, ms, tokens = got[r]
        assert ms == 200.0 and tokens == 100          # slowest rank, all tokens
        assert abs(rate - 500.0) < 1e-9               # 100 tokens / 0.2 s


def test_job_rate_single_process():
    import bench
    assert bench.job_rate(250.0, 100, 1) == (400.0, 250.0, 100)
