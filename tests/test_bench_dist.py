"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The step has no exchange between GPUs, so N ranks run N replicas; what the
ranks share is the timing: every rank times its own replica and the job is
timed by the slowest one."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    ms_local = [1.5, 2.25][rank]
    ms = bench.max_over_ranks(ms_local, "cpu")
    rate = bench.whole_job_rate(1000, ws, ms)
    q.put((rank, ms, rate, bench._dist()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate, d in res:
        assert ms == 2.25
        assert rate == pytest.approx(2 * 1000 / 2.25e-3)
        assert d[0] == 2 and d[1] == rank


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_rate(10, 1, 1.0) == 10_000.0
