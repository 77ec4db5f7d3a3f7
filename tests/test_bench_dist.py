"""The benchmark's multi-process path on CPU: two gloo ranks (127.0.0.1)
exercise the barrier and the max-over-ranks timing reduction that bench.py
uses under torchrun, and the rule that only rank 0 prints."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # each rank reports its own time; every rank must see the slowest one
        m = bench.max_over_ranks(world, 10.0 + 5.0 * rank)
        out[rank] = m
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    if not dist.is_gloo_available():
        pytest.skip("gloo not available")
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 15.0


def test_reference_arm_other_ranks_do_nothing(capsys):
    import argparse

    import bench
    args = argparse.Namespace(config="tiny", shape=None, seed=0, steps=1, warmup=3, reference_budget=1.0)
    assert bench.run_reference(args, world=2, rank=1) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank0(capsys):
    import argparse
    import json

    import bench
    args = argparse.Namespace(config="tiny", shape=None, seed=0, steps=2, warmup=3, reference_budget=1.0)
    assert bench.run_reference(args, world=1, rank=0) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["metric"] == bench.METRIC
