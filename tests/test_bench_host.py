"""Host-side logic of bench.py for N > 1 ranks, on CPU: two gloo ranks agree on
the slowest rank's step time and on the whole-job throughput; under torchrun
only rank 0 runs and prints the reference arm."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms = 2.0 + 3.0 * rank               # rank 1 is the slow one
        ms = bench.max_over_ranks(step_ms, world, "cpu")
        out.put((rank, ms, bench.job_throughput(16384, world, ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    for _, ms, value in res:
        assert ms == 5.0
        assert value == pytest.approx(2 * 16384 / 5e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_throughput(64, 1, 0.1) == pytest.approx(640000.0)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    called = []
    monkeypatch.setattr(bench, "run_reference", lambda args: called.append(args) or {})
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main()
    assert buf.getvalue() == "" and not called
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setattr(bench, "run_reference", lambda args: {"impl": "reference", "value": 1.0})
    with redirect_stdout(buf):
        bench.main()
    assert json.loads(buf.getvalue())["impl"] == "reference"
