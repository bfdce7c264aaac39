"""The N > 1 path of the benchmark, on host ranks.

Several GPUs run independent replicas of the workload: nothing is exchanged
on the data path, and the only cross-rank step is the timing reduction (a
barrier, then the maximum over ranks, so that the slowest rank sets the
time).  These tests run that step with two `gloo` ranks on the CPU and run
the reference arm under the torch launcher with two ranks, where rank 0
alone prints the result line."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # Rank r took (r + 1) * 1.5 ms: every rank must see the slowest one.
        slowest = bench._barrier_max(torch, (rank + 1) * 1.5, world)
        dist.barrier()
        # The whole-job throughput counts the work of every rank.
        calls = [{"bytes": 3_000_000, "flops": 0, "bound": "hbm"}]
        gbs = bench._throughput(calls, "GB/s", slowest * 1e-3, factor=world)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "gbs": gbs}, f)
    finally:
        dist.destroy_process_group()


def test_barrier_max_over_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for g in got:
        assert g["slowest"] == 3.0
        # 2 ranks x 3 MB in 3 ms.
        assert abs(g["gbs"] - 2.0) < 1e-12


def test_barrier_max_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench._barrier_max(torch, 4.25, 1) == 4.25


def test_reference_arm_under_launcher_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           "bench.py", "--impl", "reference", "--workload", "w4a16_tiny", "--steps", "1", "--warmup", "3",
           "--gpus", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_gpus_flag_without_launcher_starts_the_ranks():
    """`bench.py --gpus 2` run bare (no launcher in the environment) starts
    two ranks itself; rank 0 reports n_gpus = 2."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env["OMP_NUM_THREADS"] = "1"
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "w4a16_tiny", "--steps", "1",
           "--warmup", "3", "--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert json.loads(lines[0])["n_gpus"] == 2


def test_gpus_flag_must_match_the_launcher():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "w4a16_tiny", "--steps", "1",
           "--warmup", "3", "--gpus", "4"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "--gpus 4" in r.stderr
