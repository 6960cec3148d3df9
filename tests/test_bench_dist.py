"""Multi-process host logic of bench.py on CPU (gloo, world size 2).

The backward shards by rows with no exchange in the data path, so the
benchmark runs independent replicas: each rank times its own copy and the
job is as slow as its slowest rank. These checks cover that aggregation and
the reference arm's rank-0-only rule without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    my_ms = [0.020, 0.025][rank]
    slowest = bench.max_over_ranks(my_ms, ws)
    value = bench.whole_job_gbs(1e8, ws, slowest)
    out[rank] = (slowest, value)
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 0.025
    assert abs(res[0][1] - 2 * 1e8 / 25e-6 / 1e9) < 1e-6


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env.update(RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0


def test_plan_names_the_timed_kernel():
    """The bench's roofline names the row-pass kernel from the plan text of
    every backward engine."""
    sys.path.insert(0, ROOT)
    import bench
    cases = {
        "engine=row cpt=4 team_threads=128 teams=4 stages=2 grid=152 smem=131328 dw=atomic":
            "bwd_row_kernel",
        "engine=cluster csize=2 cpt=4 threads=512 stages=2 clusters=76 dw=atomic": "bwd_cluster_kernel",
        "engine=generic phase cpt=2 threads=256 grid=304 dw=atomic": "bwd_phase_kernel",
        "engine=generic realign cpb=4 rows=1 threads=512 grid=152 dw=scratch": "bwd_realign_kernel",
        "engine=generic vec rows=2 threads=512 grid=304 dw=atomic": "bwd_generic_vec_kernel",
        "engine=generic threads=512 grid=304 smem_dw=1 dw=atomic": "bwd_generic_kernel",
    }
    for plan, kernel in cases.items():
        assert bench.row_pass_kernel(plan) == kernel, plan
