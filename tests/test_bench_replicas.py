"""Host logic of the multi-process benchmark, on CPU with the gloo backend.

The GPU path does not shard across GPUs with any exchange: every rank runs an
independent replica of the workload, the step time is the maximum over ranks
and the reported throughput is all ranks' units over that time.  These tests
run two ranks as CPU processes and check exactly that host logic, plus the
clock-sample summary and the reference arm's rank-0-only output.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_info()
        assert (w, r, local) == (world, rank, rank)
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow replica
        ms_max = bench.allreduce_max(ms, w)
        bench.barrier(w)
        value = bench.whole_job_value(32768, ms_max, w)
        out_q.put((rank, ms_max, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms_max, value in got:
        assert ms_max == 15.0
        # 2 replicas x 32768 tokens in 15 ms
        assert value == pytest.approx(2 * 32768 / 0.015)


def test_whole_job_value_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.allreduce_max(3.5, 1) == 3.5
    assert bench.whole_job_value(100, 2.0, 1) == pytest.approx(50000.0)


def test_clock_summary_uses_samples_inside_the_region():
    sys.path.insert(0, ROOT)
    import bench
    c = bench.Clocks(0)
    c.t_open, c.t_close = 10.0, 10.5
    c.lines = [(9.0, "900, 2070, 300, Not Active, Not Active, Not Active, Not Active\n"),
               (10.2, "2070, 2070, 900, Not Active, Not Active, Not Active, Active\n"),
               (10.4, "2055, 2070, 950, Not Active, Not Active, Not Active, Not Active\n"),
               # half a sampling period after the region closed: it still covers the end
               (10.5 + bench.Clocks.PERIOD_MS / 2000,
                "2040, 2070, 950, Not Active, Not Active, Not Active, Not Active\n"),
               (12.0, "600, 2070, 100, Active, Not Active, Not Active, Not Active\n")]
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2055.0
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_short_region_takes_the_nearest_sample():
    sys.path.insert(0, ROOT)
    import bench
    c = bench.Clocks(0)
    c.t_open, c.t_close = 10.0, 10.01
    c.lines = [(9.95, "2070, 2070, 900, Not Active, Not Active, Not Active, Not Active\n"),
               (12.0, "1000, 2070, 900, Not Active, Not Active, Not Active, Not Active\n")]
    s = c.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 2070.0 and s["reasons"] == []
    c.lines = []
    assert bench.Clocks(0).summary()["reasons"] == ["unsampled"]


def _reference_rank(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup = 1, 0
    buf = io.StringIO()
    with redirect_stdout(buf):
        if rank == 0:
            # rank 0 would time the oracle; only check that rank 1 prints nothing
            out_q.put((rank, "skipped"))
            return
        bench.reference_main(A, world, rank)
    out_q.put((rank, buf.getvalue()))


def test_reference_arm_prints_only_on_rank_zero():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_reference_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    assert got[1] == ""


def test_reference_arm_line_on_rank_zero(monkeypatch):
    """The reference arm's JSON line carries the keys the harness reads."""
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    oracle.build()

    class A:
        steps, warmup = 1, 0
    # a smaller oracle step keeps this CPU test fast; the code path is the same
    monkeypatch.setattr(bench, "REFERENCE_STEP", dict(tokens=128, heads=2))
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference_main(A, 1, 0)
    line = json.loads(buf.getvalue())
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "cpu_baseline", "e2e", "config", "dtype"):
        assert key in line
    assert line["impl"] == "reference"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["value"] > 0
