"""Replica runs of bench.py (one process per GPU, no collective on the data path): the
cross-rank reduction of the step time and the whole-job rate, checked with two gloo ranks on
CPU; the reference arm runs on rank 0 only."""
import os
import socket
import sys
import time

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = [2.0, 5.0][rank]  # rank 1 is the slow replica
        ms, value = bench.whole_job(ms_local, 32768, world, torch.device("cpu"))
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_whole_job_rate_two_replicas():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=120)
        assert pr.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, value in got:
        assert ms == 5.0  # the slowest rank's step time on every rank
        assert value == pytest.approx(2 * 32768 / 5e-3 / 1e6)


def test_whole_job_rate_one_process():
    ms, value = bench.whole_job(4.0, 1000, 1)
    assert ms == 4.0 and value == pytest.approx(1000 / 4e-3 / 1e6)


def test_reference_arm_runs_on_rank_zero_only():
    class A:
        steps, warmup = 1, 0
    assert bench.run_reference(A(), rank=1) is None


def test_reference_arm_reports_our_arm_config(monkeypatch):
    """The reference arm's line names the same workload as ours (same metric, unit and config);
    only the timing note and the statement of the per-step sample differ. The oracle step itself
    is replaced here: this checks the line."""
    monkeypatch.setattr(bench, "_oracle_step", lambda p, f, cores: time.sleep(0.001))

    class A:
        steps, warmup, tokens, mode = 2, 1, 32768, "exact"
    res = bench.run_reference(A(), rank=0)
    ours = bench.workload_config(32768, 8, 2, "exact", True, True)
    assert res["impl"] == "reference" and res["metric"] == bench.METRIC and res["unit"] == bench.UNIT
    own = ("l2", "sample_tokens_per_step", "sample")
    assert {k: v for k, v in res["config"].items() if k not in own} == {k: v for k, v in ours.items() if k != "l2"}
    assert res["config"]["sample_tokens_per_step"] == 1024 and "1024" in res["config"]["sample"]
    assert res["cpu_baseline"]["kind"] == "oracle" and res["e2e"]["h2d_bytes_per_step"] == 0
