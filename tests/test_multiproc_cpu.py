"""Host-side logic of the multi-GPU benchmark path, run as world-size-2 gloo
process groups on the CPU (the workload is replicated per GPU: no data-path
collective, only the barrier and the max over ranks of the timings), and the
reference arm's JSON line."""
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
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w, _ = bench.dist_init(world)
    bench.barrier(w)
    ms_max = bench.max_over_ranks(10.0 * (r + 1), w)          # rank 1 is the slow one
    value = bench.job_throughput(1e9, 4, w, ms_max)
    with open(os.path.join(out_dir, "rank%d.json" % r), "w") as f:
        json.dump({"rank": r, "world": w, "ms_max": ms_max, "value": value,
                   "backend": dist.get_backend()}, f)
    dist.destroy_process_group()


def test_two_rank_gloo_max_and_throughput(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(2)]
    for r in res:
        assert r["world"] == 2 and r["backend"] == "gloo"
        assert r["ms_max"] == 20.0                            # max over ranks, seen by every rank
        # 2 ranks x 4 steps x 1 GB over 20 ms
        assert abs(r["value"] - 2 * 4 * 1e9 / 20e-3 / 1e9) < 1e-9


def test_reference_arm_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "0"], capture_output=True, text=True, env=env, timeout=600)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["metric"].startswith("quant-matmul weight GB/s")


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1"],
                         capture_output=True, text=True, env=env, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == ""
