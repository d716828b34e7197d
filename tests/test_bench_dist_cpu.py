"""CPU (gloo) tests of bench.py's multi-process path, world_size 2.

The path shards into independent replicas: the only collectives are the barrier before
the timed region and the maximum of the ranks' times. Both run here on CPU ranks over gloo,
as does the reference arm under torchrun (rank 0 prints the one JSON line, the other rank
exits 0 without work).
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    import bench
    dist.barrier()
    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.25 * rank], world, "cpu")
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump(got, f)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    for r in range(world):
        with open(tmp_path / ("rank%d.json" % r)) as f:
            assert json.load(f) == [2.0, 10.0, 0.25]


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3, 1.5], 1, "cpu") == [3.0, 1.5]


def test_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="4")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] > 0
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["e2e"]["d2h_bytes_per_step"] == 0
    assert res["cpu_baseline"]["kind"] == "oracle"
