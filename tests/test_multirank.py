"""Multi-process (gloo, world size 2, CPU) test of bench.py's N>1 host logic: every rank runs its
own replica, the step time is the maximum over ranks, and the reported value aggregates all
ranks' work (weak scaling).  No data-path collective exists."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench._dist()
        assert (w, r, lr) == (world, rank, rank)
        bench._barrier(world)
        t = 1.0 + rank                           # rank 1 is the slow one
        t_max = bench._max_over_ranks(t, world, torch.device("cpu"))
        v = bench.aggregate_value(world, 21.762e9, t_max)
        q.put((rank, t_max, v, bench.rank_seed(1002, rank)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [t for _, t, _, _ in res] == [2.0, 2.0]                 # both see the slowest rank
    assert res[0][2] == pytest.approx(2 * 21.762e9 / 2e-3 / 1e12)  # whole-job work / job time
    assert res[0][3] != res[1][3]                                  # independent replicas


def test_gpus_flag_launches_one_process_per_gpu(monkeypatch):
    """`bench.py --gpus N` outside a launcher relaunches itself under torch.distributed.run with N
    processes; inside one, a WORLD_SIZE that disagrees with --gpus is refused."""
    import bench
    seen = []
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: seen.append(cmd) or 0)
    assert bench.main(["--gpus", "4", "--steps", "7", "--warmup", "3"]) == 0
    cmd = seen[0]
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"]
    assert cmd[cmd.index("--nproc-per-node") + 1] == "4"
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-6:] == ["--gpus", "4", "--steps", "7", "--warmup", "3"]
    monkeypatch.setenv("WORLD_SIZE", "3")
    assert bench.main(["--gpus", "2"]) == 2
