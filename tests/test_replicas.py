"""Multi-process pieces of the benchmark on CPU (gloo, world size 2).

The path shards only as independent replicas: no collective touches the data,
only the timed region's length is combined (max over ranks), and the reference
arm runs on rank 0 alone.
"""
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


def _worker(rank, world, port, values, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = bench.max_over_ranks(values[rank])
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        values = [3.5, 7.25]
        procs = [ctx.Process(target=_worker, args=(r, 2, port, values, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == out[1] == 7.25


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks(4.0) == 4.0


def test_reference_arm_skips_other_ranks(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), dict(steps=1, warmup=0, layers=0, tokens=0, gpus=2))()
    bench.run_reference(args, bench.config_by_name("opt7b_stack"))
    assert capsys.readouterr().out == ""
