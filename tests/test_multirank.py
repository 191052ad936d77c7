"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The projection shards by token rows with no exchange step, so several GPUs run
independent replicas; what needs testing is the host side: every rank joins
the barrier, the whole-job time is the slowest rank's, the units are summed
over ranks, and only rank 0 prints.  These run as gloo process groups on CPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank), "BENCH_DIST_BACKEND": "gloo"})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    # rank r "took" 10 + 5 r ms and processed 1000 (r + 1) units
    ms, units, per_s = bench.aggregate(10.0 + 5.0 * r, 1000.0 * (r + 1), w)
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"ms": ms, "units": units, "per_s": per_s}, f)
    dist.destroy_process_group()


def test_aggregate_two_ranks_gloo(tmp_path):
    world = 2
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:  # every rank sees the same whole-job figures
        assert r["ms"] == 15.0  # the slowest rank's time
        assert r["units"] == 3000.0  # units of all ranks
        assert r["per_s"] == pytest.approx(3000.0 / 15e-3)


def test_aggregate_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.aggregate(4.0, 8.0, 1) == (4.0, 8.0, 2000.0)


def test_reference_arm_under_torchrun_prints_one_line():
    """torchrun with 2 ranks: rank 0 alone times the oracle and prints one JSON
    line; rank 1 exits 0 without work."""
    env = dict(os.environ, BENCH_DIST_BACKEND="gloo", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3", "--cpu-seconds", "1"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] == d["cpu_baseline"]["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
