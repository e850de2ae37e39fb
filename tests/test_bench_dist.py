"""bench.py's multi-process path on CPU (gloo, world size 2): the ranks are replicas, so the only
collectives are the barrier around the timed region and the reductions of the result (the slowest
rank's time, every rank's commits).  The reference arm runs on rank 0 alone."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank), SPD_DIST_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    ws, r, local = bench.dist_setup(None)
    ms = 100.0 + 50.0 * r              # rank 1 is the slower one
    commits = 10.0 * (r + 1)
    bench.barrier(ws)
    ms_max = bench.allreduce(ms, bench._max_op(), ws)
    commits_all = bench.allreduce(commits, bench._sum_op(), ws)
    bench.barrier(ws)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump(dict(ws=ws, rank=r, local=local, ms_max=ms_max, commits_all=commits_all,
                       value=bench.job_value(ms_max, commits_all)), f)
    dist.destroy_process_group()


def test_two_replicas_reduce_time_by_max_and_commits_by_sum(tmp_path):
    mp.start_processes(_worker, args=(_free_port(), str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert (d["ws"], d["rank"], d["local"]) == (2, r, r)
        assert d["ms_max"] == 150.0          # the slowest rank's time
        assert d["commits_all"] == 30.0      # every rank's commits
        assert d["value"] == pytest.approx(30.0 / 0.150)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    called = []
    monkeypatch.setattr(bench, "oracle_sample", lambda *a, **k: called.append(1))

    class A:
        steps, warmup, mode = 4, 1, "forced-0.6"
    assert bench.main_reference(A, 2, 1) is None
    assert called == []                      # rank 1 does no work and prints nothing
