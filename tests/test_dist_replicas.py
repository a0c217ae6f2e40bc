"""Multi-process host logic of bench.py's replica mode (CPU, gloo, two ranks):
the timed region's duration is the maximum over ranks, and the whole-job
value counts every rank's work over that time.  The attention path itself
runs independent replicas (no collective on the data path)."""

import json
import os
import socket
import tempfile

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"))
        value = bench.job_tflops(2.0e12, ms, world)
        with open(os.path.join(outdir, f"r{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_with_two_gloo_ranks():
    world = 2
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_worker, args=(world, _free_port(), d), nprocs=world, join=True)
        res = [json.load(open(os.path.join(d, f"r{r}.json"))) for r in range(world)]
    for r in res:
        assert r["ms"] == pytest.approx(15.0)
        # 2 ranks x 2e12 flops in 15 ms
        assert r["value"] == pytest.approx(2 * 2.0e12 / 0.015 / 1e12)


def test_single_process_is_its_own_max():
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.job_tflops(1e12, 1000.0, 1) == pytest.approx(1.0)


def test_reference_arm_prints_only_on_rank_zero(capsys, monkeypatch):
    class A:
        ref_sample_L = 64
        warmup = 0
        steps = 1
        workload = bench.DEFAULT
    bench.run_reference(A, bench.WORKLOADS[bench.DEFAULT], world=2, rank=1)
    assert capsys.readouterr().out == ""
    bench.run_reference(A, bench.WORKLOADS[bench.DEFAULT], world=2, rank=0)
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
