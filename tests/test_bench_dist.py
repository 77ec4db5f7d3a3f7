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


def test_weight_banks_keep_every_step_in_hbm():
    """Workloads whose active weights fit in L2 rotate over enough copies of
    the expert banks that the copies' active weights exceed three times the
    L2; the others use one bank."""
    import bench
    from mixture_experts_expert_router_gb300 import workloads as W

    class Shape:
        def __init__(self, T, H, I, E, k):
            self.T, self.H, self.I, self.num_local, self.top_k = T, H, I, E, k

    for name in ("decode_t1", "decode_t8", "decode_t64", "prefill_few_large", "prefill_many_fine"):
        c = W.MOE_CONFIGS[name]
        s = Shape(c["T"], c["H"], c["I"], c["E"], c["top_k"])
        active = min(s.num_local, s.T * s.top_k) * 3 * s.H * s.I * 2
        n = bench.weight_banks(s)
        if active >= 3 * bench.L2_NOMINAL:
            assert n == 1, name
        else:
            assert n * active >= 3 * bench.L2_NOMINAL and (n - 1) * active < 3 * bench.L2_NOMINAL, name
    assert bench.weight_banks(Shape(1, 2048, 768, 128, 8)) == 6  # 8 experts x 9.4 MB


def test_bench_accounting_matches_published_targets():
    """The benchmark's algorithmic FLOPs and bytes for the default workload
    (8 experts, all active; logits routing) equal the target table's
    2.886 TFLOP and 2.886 GB, and the decode T=1 bytes (8 distinct experts,
    pre-routed) its 75.5 MB."""
    import numpy as np
    import bench

    class Shape:
        def __init__(self, T, H, I, E, k, mode):
            self.T, self.H, self.I, self.E, self.top_k, self.mode = T, H, I, E, k, mode
            self.num_local, self.local_offset = E, 0

    wl = Shape(4096, 4096, 14336, 8, 2, "logits")
    ids = np.tile(np.arange(8, dtype=np.int32), 4096 * 2 // 8)
    F = bench.layer_flops(len(ids), wl.H, wl.I)
    B, active = bench.layer_bytes(wl, ids)
    assert active == 8
    assert abs(F / 1e12 - 2.886) < 0.0005
    assert abs(B / 1e9 - 2.886) < 0.0005
    wl = Shape(1, 2048, 768, 128, 8, "prerouted")
    B, active = bench.layer_bytes(wl, np.array([3, 9, 17, 40, 41, 77, 100, 127], np.int32))
    assert active == 8 and abs(B / 1e6 - 75.5) < 0.05


def test_recorded_traffic_follows_every_source(tmp_path, monkeypatch):
    """profiles/traffic.json: a stage's bytes are attached only while every
    kernel source it lists still has the recorded hash."""
    import hashlib
    import json

    import bench
    (tmp_path / "profiles").mkdir()
    a, b = tmp_path / "a.cu", tmp_path / "b.cu"
    a.write_text("kernel a")
    b.write_text("kernel b")
    sha = lambda p: hashlib.sha256(p.read_bytes()).hexdigest()[:16]
    rec = {"captures": [{"workload": "w", "kernel": "fc1_swiglu", "bytes": 123, "sources": ["a.cu", "b.cu"],
                         "sources_sha16": [sha(a), sha(b)]}]}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("w", "fc1_swiglu") == 123
    assert bench.recorded_traffic("w", "fc2") is None
    assert bench.recorded_traffic("other", "fc1_swiglu") is None
    b.write_text("kernel b, changed")
    assert bench.recorded_traffic("w", "fc1_swiglu") is None

