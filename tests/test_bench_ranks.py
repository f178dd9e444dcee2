"""The bench's multi-rank logic on CPU with two gloo ranks: every rank runs a
replica, the timed duration is the maximum over ranks, and only rank 0 reports."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        elapsed = 10.0 + 5.0 * rank                 # rank 1 is the slowest replica
        results[rank] = bench.max_over_ranks(elapsed, world)
        # the reference arm does its work on rank 0 only
        args = bench.parse_args(["--impl", "reference"])
        if rank != 0:
            assert bench.run_reference(args, rank, world) is None
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world, join=True,
                       start_method="spawn")
    assert results[0] == results[1] == 15.0


def test_dist_env_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("LOCAL_RANK", "3")
    assert bench.dist_env() == (3, 4, 3)


def test_bench_argument_defaults():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "ours" and a.warmup >= 3
    assert a.workload == "llama3.1-8b-decode-layer"


def test_reference_arm_line_on_cpu(capsys, monkeypatch):
    """The reference arm (the oracle on host cores) prints one JSON line with
    the contract's keys on the small exact workload; it needs no GPU."""
    import json
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.main(["--impl", "reference", "--workload", "tiny_exact", "--steps", "2", "--warmup", "3",
                       "--ref-tokens", "1024"]) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["n_gpus"] == 1 and d["higher_is_better"]
    assert d["value"] > 0 and d["steps"] == 2 and d["config"]["seq_len"] == 1024
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
