"""Multi-process form of the benchmark (independent replicas: the renderer
has no exchange step) on CPU with the gloo backend, world size 2: every rank renders its own frame,
the only collective is the max over ranks of the timed region, and only
rank 0 reports.  No GPU."""
from __future__ import annotations

import json
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    w, r, local = bench.dist_env()
    # rank r "took" 10 + r ms: the job's time is the slowest rank's
    total = bench.max_over_ranks(10.0 + r, dist, "cpu")
    rate = bench.job_rate(w, 6, 5, total)
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, w, local, total, rate))


def test_two_replicas_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    assert [o[2] for o in out] == [0, 1]
    for _, _, _, total, rate in out:
        assert total == 11.0
        # both replicas' camera frames (2 x 6 x 5 steps) over the slowest rank's time
        assert rate == pytest.approx(2 * 6 * 5 / 0.011)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_rate(1, 1, 10, 5.0) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    """Under torchrun the reference arm (the oracle on host cores) runs once:
    ranks other than 0 return at once, printing nothing."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference"])
    bench.run_reference(bench.args_parse())
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_contract_line(capsys, monkeypatch):
    """Rank 0 of the reference arm times the oracle on the host cores and
    prints one JSON line with the keys the bench contract names (a one-second
    sample here)."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1",
                                      "--warmup", "0", "--cpu-seconds", "1"])
    bench.run_reference(bench.args_parse())
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is True and line["value"] > 0
    assert line["ms_per_step"] == pytest.approx(1e3 / line["value"])
    assert line["steps"] == 1 and line["warmup"] == 0 and line["n_gpus"] == 1
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
