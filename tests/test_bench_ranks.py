"""bench.py on more than one rank, on CPU ranks over gloo (world size 2): the whole-job
aggregation (the slowest rank's time, every rank's rows, rows/s over all of them), the barrier,
and the reference arm launched by torchrun, where rank 0 alone runs and prints its JSON line
and the other rank exits 0 without work. The GPU arm's timed region needs a GPU;
what it hands to this aggregation is what is tested here."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    # CPU ranks over gloo even where a GPU is present (CUDA initialises lazily)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w, _ = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    # rank 0 timed 2 ms for 300 rows, rank 1 timed 5 ms for 500 rows
    ms, rows, value = bench.whole_job([2.0, 5.0][r], [300, 500][r], w)
    out[r] = (ms, rows, value)
    dist.destroy_process_group()


def test_whole_job_over_two_ranks():
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(2, free_port(), out), nprocs=2, join=True)
    for r in range(2):
        ms, rows, value = out[r]
        assert ms == 5.0 and rows == 800
        assert value == pytest.approx(800 / 5e-3)


def test_whole_job_single_rank_is_local():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job(4.0, 1000, 1) == (4.0, 1000, pytest.approx(250000.0))


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1",
           "--workload", "tiny_greedy"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")       # CPU ranks over gloo
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["config"]["workload"] == "tiny_greedy"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
