"""The benchmark's multi-rank path on CPU: two ranks over gloo (127.0.0.1).

Each replica times its own GEMMs; the only cross-rank steps are a barrier
around the timed region and a max-reduce of its duration.  The reference arm
runs and prints on rank 0 alone; the other ranks exit 0 without work."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

torch = pytest.importorskip("torch")


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    args = argparse.Namespace(impl="reference")
    w, r, local = bench.dist_setup(args)
    bench.barrier(w)
    got = bench.max_over_ranks(1.5 + 10.0 * rank, w)
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "local": local, "max": got}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max_reduce(tmp_path):
    import torch.multiprocessing as mp
    port = free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert d["world"] == 2 and d["rank"] == r and d["local"] == r
        assert d["max"] == pytest.approx(11.5)  # the slowest replica's time is the job's


def test_reference_arm_prints_on_rank_zero_only():
    env_base = dict(os.environ, WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", MASTER_PORT=str(free_port()))
    outs = []
    for rank in (0, 1):
        env = dict(env_base, RANK=str(rank), LOCAL_RANK=str(rank))
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                            "--workload", "bf16_256", "--steps", "1", "--warmup", "3", "--ref-step-s", "0.05"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append([ln for ln in r.stdout.splitlines() if ln.startswith("{")])
    assert len(outs[0]) == 1 and outs[1] == []
    line = json.loads(outs[0][0])
    assert line["impl"] == "reference" and line["value"] > 0
    for key in ("metric", "unit", "n_gpus", "steps", "warmup", "cpu_baseline", "e2e", "config"):
        assert key in line


def test_gpus_flag_relaunches_one_process_per_replica():
    # --gpus 2 outside torchrun: the script relaunches itself under torchrun with two ranks
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "bf16_256", "--steps", "1", "--warmup", "3", "--ref-step-s", "0.05"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2


def test_gpus_flag_disagreeing_with_the_launcher_is_refused():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "bf16_256", "--steps", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 2 and "WORLD_SIZE" in r.stderr
