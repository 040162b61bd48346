"""The replicas-only multi-GPU path of the benchmark, checked on the CPU with two
gloo ranks (no GPU): every rank runs the same independent (batch, kv-head)
work, the step time is the slowest rank's, the whole-job value counts the work
of all ranks over that time, and the reference arm prints from rank 0 alone.
"""
import contextlib
import io
import json
import os
import socket
import sys
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(torch, dist, local_ms[rank], world)
        value = bench.whole_job_tflops(world, 1.0e12, 10, slowest)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "value": value}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_work(tmp_path):
    world, port = 2, _free_port()
    local_ms = [120.0, 150.0]  # rank 1 is the slow one
    mp.start_processes(_rank_main, args=(world, port, local_ms, str(tmp_path)), nprocs=world, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["slowest"] == 150.0
        # two ranks x 10 steps x 1 TFLOP each over 150 ms
        assert r["value"] == pytest.approx(2 * 10 * 1.0 / 0.150)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(torch, None, 7.5, 1) == 7.5
    assert bench.whole_job_tflops(1, 2.0e12, 4, 8.0) == pytest.approx(4 * 2.0 / 0.008)


def test_reference_arm_prints_from_rank_zero_only(monkeypatch):
    pytest.importorskip("oracle")
    from causal_gqa_flash_gb300.inputs import WORKLOADS
    args = types.SimpleNamespace(gpus=2, steps=1, warmup=0)
    w = WORKLOADS["c1"]
    for rank, expect_line in ((1, False), (0, True)):
        monkeypatch.setenv("RANK", str(rank))
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            assert bench.run_reference(args, w) == 0
        lines = [l for l in buf.getvalue().splitlines() if l.startswith("{")]
        if expect_line:
            assert len(lines) == 1
            d = json.loads(lines[0])
            assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
        else:
            assert lines == []
