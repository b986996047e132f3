"""The N > 1 path of bench.py on the CPU: world-size-2 `gloo` process groups.

On N GPUs the bench runs N independent replicas of the sweep (the path has no
exchange step, so no data-path collective).  What it does across ranks is host
logic, tested here without a GPU:

* the timed region ends when the slowest replica ends (all-reduce MAX);
* the whole-job rate counts every rank's steps within that time (weak
  scaling);
* under `--impl reference` only rank 0 runs and prints; the other ranks exit
  0 without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

from conftest import ROOT

torch = pytest.importorskip("torch")
import torch.distributed as dist          # noqa: E402
import torch.multiprocessing as mp        # noqa: E402

sys.path.insert(0, ROOT)
import bench                             # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, local_ms, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        env_ws, env_rank, env_local = bench.dist_env()
        assert (env_ws, env_rank, env_local) == (ws, rank, rank)
        dist.barrier()
        ms = bench.max_over_ranks(torch, local_ms[rank], ws, torch.device("cpu"))
        value, tok = bench.job_rates(1_000_000_000, 10, ws, ms)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value, "tok": tok}, f)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("local_ms", [[12.5, 20.0], [33.0, 7.25]])
def test_two_gloo_ranks_take_the_slowest_time(tmp_path, local_ms):
    ws = 2
    mp.start_processes(_rank_main, args=(ws, free_port(), local_ms, str(tmp_path)), nprocs=ws, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(ws)]
    slowest = max(local_ms)
    for r in res:
        assert r["ms"] == slowest
        # 10 steps of 1 GB on each of 2 ranks within the slowest rank's time
        assert r["value"] == pytest.approx(2 * 10 * 1.0 / (slowest * 1e-3))
        assert r["tok"] == pytest.approx(2 * 10 / (slowest * 1e-3))


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(torch, 4.5, 1, torch.device("cpu")) == 4.5
    v1, t1 = bench.job_rates(16_174_817_280, 400, 1, 1732.0)
    v2, t2 = bench.job_rates(16_174_817_280, 400, 2, 1732.0)
    assert v2 == pytest.approx(2 * v1) and t2 == pytest.approx(2 * t1)


def test_reference_arm_non_zero_rank_prints_nothing():
    # rank 1 of 2 of `--impl reference` leaves before any work: no oracle run, no output
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_gpus_must_match_the_launched_ranks():
    # --gpus 2 in a single process (no torchrun) is an error, not one silent replica
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "3",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "WORLD_SIZE=1" in r.stderr
