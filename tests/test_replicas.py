"""The N > 1 path of bench.py on the CPU: two gloo ranks on 127.0.0.1.

The path has no exchange step, so the replicas share only host-side
coordination: a barrier before the timed region, the maximum of the timed
region over ranks (the slowest replica sets the job's time), a whole-job value
= every rank's bytes over that time, and a single report from rank 0. The
reference arm does its work on rank 0 only."""
import json
import multiprocessing as mp
import os
import socket
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    rep = bench.Replicas()
    rep.barrier()
    ms = rep.max_over_ranks(10.0 + 5.0 * rank)  # rank 1 is the slower replica
    value = rep.job_value(2.0e9, ms)
    args = type("A", (), {"steps": 1, "warmup": 0})()
    ref = bench.run_reference(args) if rank != 0 else "skipped"
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"world": rep.world, "ms": ms, "value": value, "reports": rep.reports,
                   "ref_is_none": ref is None}, f)
    rep.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas(tmp_path):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["world"] == 2
        assert r["ms"] == pytest.approx(15.0)  # max over ranks
        # 2 ranks x 2 GB per step in 15 ms
        assert r["value"] == pytest.approx(2 * 2.0e9 / 15e-3 / 1e9)
    assert res[0]["reports"] and not res[1]["reports"]
    assert res[1]["ref_is_none"]  # the reference arm runs on rank 0 only


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench

    rep = bench.Replicas()
    assert rep.world == 1 and rep.reports
    rep.barrier()
    assert rep.max_over_ranks(3.5) == 3.5
    assert rep.job_value(1.0e9, 1.0) == pytest.approx(1000.0)


def test_gpus_flag_launches_its_own_replicas():
    """bench.py --gpus 2 without torchrun starts two processes itself (ranks 0 and
    1 over gloo on 127.0.0.1); only rank 0 prints, with n_gpus = 2."""
    import subprocess

    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "LOCAL_RANK", "WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--replica-selftest"],
                       capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line == {"n_gpus": 2, "max_over_ranks": 2.0}
