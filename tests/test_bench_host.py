"""Host-side logic of bench.py: max-over-ranks timing with world_size 2 (gloo), and
the reference arm's output line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.aggregate_over_ranks(torch, dist, 10.0 + 5.0 * rank)
    q.put((rank, got))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 15.0, 1: 15.0}


def test_single_process_aggregation_is_identity():
    assert bench.aggregate_over_ranks(torch, None, 3.5) == 3.5


def test_reference_arm_line(monkeypatch, capsys):
    monkeypatch.setattr(bench, "ORACLE_SAMPLE", (1, 64))
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == bench.UNIT and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1"]) == 0
    assert capsys.readouterr().out == ""
