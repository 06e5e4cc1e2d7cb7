"""The benchmark's N > 1 path on CPU: two gloo ranks (no GPU).

Each rank runs the whole workload on its own GPU in a real run (weak scaling, no collective on
the data path); the only exchange is the maximum of the per-rank times. These tests run that
host logic with world_size 2 over gloo."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = [12.5, 10.0][rank]                       # rank 0 is the slow one
    mx = bench.reduce_max(elapsed)
    val = bench.job_value(1_000_000_000, 4, mx, world)
    dist.barrier()
    q.put((rank, mx, val))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [12.5, 12.5]
    # 2 ranks x 1 GB x 4 steps over 12.5 ms
    assert all(abs(r[2] - 2 * 4 / 12.5e-3) < 1e-6 for r in res)


def test_reference_arm_only_rank0_works(monkeypatch, capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        workload, steps, warmup, ref_step_seconds = "cfg1", 1, 0, 0.1
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
