"""The replicas-only multi-rank logic of bench.py on CPU: two gloo ranks.

Each GPU runs an independent replica of the hot path on its own seeded
input, so the only cross-rank step is host bookkeeping: the job's throughput
is the units all ranks processed divided by the slowest rank's time, and the
reference arm runs on rank 0 alone."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    w, r, _ = bench.dist_setup(None)
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    # rank r processed (r + 1) * 1000 units in (r + 1) * 10 ms
    value, ms = bench.job_throughput((rank + 1) * 1000, (rank + 1) * 10.0, w)
    bench.barrier(w)
    q.put((rank, value, ms))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_job_throughput_is_sum_over_max(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    units = sum((r + 1) * 1000 for r in range(world))
    ms = world * 10.0
    for _, value, got_ms in res:
        assert got_ms == ms
        assert value == pytest.approx(units / (ms / 1e3))


def test_single_rank_is_local():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.job_throughput(500, 20.0, 1)
    assert ms == 20.0 and value == pytest.approx(25000.0)


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup = 1, 3
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
