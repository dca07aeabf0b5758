"""The N > 1 path of bench.py: every rank runs an independent replica (the
model does not shard), the timed region is closed by a barrier and the job's
time is the slowest rank's. Exercised here with two gloo ranks on the CPU."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    elapsed = [2.0, 3.5][rank]           # rank 1 is the slow one
    value, t = bench.aggregate_throughput(128 * 10, elapsed, world)
    out[rank] = (value, t, bench.max_over_ranks(float(rank), world))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        value, t, mx = out[rank]
        assert t == pytest.approx(3.5)
        assert value == pytest.approx(128 * 10 * world / 3.5)
        assert mx == 1.0


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
