"""The benchmark's multi-rank path on the CPU (gloo, world size 2, 127.0.0.1):
replicas only, so the only collective is the max over ranks of the timed region;
the whole-job value counts every rank's replica; only rank 0 runs the reference
arm.  No GPU is needed: the device-side work is not part of what is tested."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        assert bench.rank_env() == (world, rank, rank)
        mine = 10.0 + 7.5 * rank  # each rank's own timed region (ms)
        got = bench.max_over_ranks(mine, dist, "cpu")
        value = bench.whole_job_tflops(2.0e12, 4, world, got)
        out.put((rank, got, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_and_count_both_replicas():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(out.get(timeout=10) for _ in range(world))
    slowest = 10.0 + 7.5 * (world - 1)
    for rank, got, value in res:
        assert got == pytest.approx(slowest)
        # two replicas of 4 steps of 2 TFLOP each in the slowest rank's 17.5 ms
        assert value == pytest.approx(world * 2.0e12 * 4 / (slowest / 1e3) / 1e12)


def test_single_process_is_its_own_maximum():
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5
    assert bench.whole_job_tflops(1e12, 2, 1, 1000.0) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    class A:
        workload, steps, warmup = "tiny_1x1x256x32", 1, 0

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A())
    assert buf.getvalue() == ""
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A())
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["dtype"] == "f64"
    # the sample is rows 0..255 of the 256-row workload: 14 n^2 d / 2 FLOPs counted
    assert "0..255" in line["cpu_baseline"]["sample"]
