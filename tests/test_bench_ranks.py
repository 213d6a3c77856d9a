"""The multi-process path of bench.py on CPU (no GPU): with N replicas, one
process per GPU, the job's time is the slowest rank's (max over ranks), and
under torchrun only rank 0 runs and prints the reference arm, whose line
keeps the GPU arm's metric, unit and config."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(torch, 10.0 * rank + 1.5)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_time_is_the_slowest_rank_with_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert got == [(0, 11.5), (1, 11.5)]


def test_single_process_time_is_unchanged():
    assert bench.max_over_ranks(torch, 3.25) == 3.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    """Rank 0 (no torchrun) times the fp64 oracle on a bounded sample of one
    step and prints one JSON line with the GPU arm's metric, unit and config
    (about 15 s: the mixed workload is built and one step is sampled)."""
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1"]) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "us" and line["higher_is_better"] is False
    assert line["steps"] == 1 and line["warmup"] >= 3 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["ms_per_step"] == pytest.approx(line["value"] / 1e3, rel=1e-3)
    assert line["dtype"] == "f64" and "mixed continuous-batching step" in line["config"]["workload"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "us", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
