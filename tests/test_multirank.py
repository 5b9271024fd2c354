"""Multi-rank logic of bench.py on the CPU (gloo, world size 2).

The quantize path shards by rows and needs no exchange, so N GPUs run N
independent replicas; what is shared between ranks is only the timing: the
whole-job rate is every rank's bytes over the slowest rank's time, and the
reference arm (the CPU oracle) runs on rank 0 alone.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env()[:2] == (world, rank)
        # rank r took 1 + r seconds for 10 steps of 100 units each
        t_max, rate = bench.job_throughput(1.0 + rank, world, 100.0, 10)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"t_max": t_max, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_job_throughput_takes_slowest_rank(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        got = json.load(open(tmp_path / f"rank{r}.json"))
        assert got["t_max"] == 2.0
        assert got["rate"] == world * 100.0 * 10 / 2.0


def test_job_throughput_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(0.5, 1, 8.0, 4) == (0.5, 64.0)


def _run_reference(rank, world, extra=()):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--gpus", str(world), "--steps", "1", "--warmup", "0",
                           "--oracle-rows", "2", *extra],
                          env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_only_rank0_prints():
    r1 = _run_reference(1, 2)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run_reference(0, 2)
    assert r0.returncode == 0, r0.stderr
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
