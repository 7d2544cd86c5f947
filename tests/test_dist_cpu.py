"""The multi-process path of bench.py on CPU with gloo (world size 2): each
rank runs its own replica, the timed region's end is the slowest rank's, and
the whole-job rate counts every rank's tokens.  No GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [12.5, 30.0][rank]                       # rank 1 is the slow one
    ms = bench.reduce_max(local_ms)
    rate = bench.whole_job_rate(4096, world, 10, ms / 1e3)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"ms": ms, "rate": rate}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_rate(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    r0 = json.load(open(tmp_path / "r0.json"))
    r1 = json.load(open(tmp_path / "r1.json"))
    assert r0["ms"] == r1["ms"] == 30.0                  # max over ranks
    assert r0["rate"] == pytest.approx(4096 * 2 * 10 / 0.030)


def test_reduce_max_without_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.25) == 3.25
    assert bench.whole_job_rate(4096, 1, 2, 0.5) == 4096 * 2 / 0.5


def test_reference_arm_rank1_does_nothing():
    """Under torchrun the reference arm runs on rank 0 only: another rank
    exits 0 without output."""
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line(orc):
    """Rank 0 of the reference arm prints one JSON line with the oracle's
    rate and the keys the driver reads."""
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.5"], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == len(os.sched_getaffinity(0))
    assert cb["single_thread_value"] > 0 and cb["nproc"] == os.cpu_count()
    assert line["e2e"]["h2d_bytes_per_step"] == 0
