"""Multi-process host logic of bench.py on CPU (gloo, world size 2): the
max-over-ranks reduction of the timed regions, the whole-job throughput of
independent replicas, and the reference arm's single output line under
torchrun.  The step shards by request with no exchange, so these are the only
multi-rank paths (replicas only)."""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    q.put((rank, bench.max_over_ranks(1.5 + rank, "cpu", ws)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 2.5, 1: 2.5}


def test_replica_throughput_counts_every_rank():
    import bench
    assert bench.max_over_ranks(3.25, "cpu", 1) == 3.25
    # 4 ranks, 100 verifies each, slowest rank 50 ms -> 8000 verifies/s for the job
    assert abs(bench.replica_throughput(100, 50.0, 4) - 8000.0) < 1e-9


def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny", "--steps", "1", "--warmup", "0",
           "--cpu-budget-s", "2"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "verifies/s"
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"] == {"value": d["value"], "unit": "verifies/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_tree_option_builds_the_requested_trees():
    import argparse

    import bench
    a = argparse.Namespace(workload="vicuna7b", tree=None)
    assert len(bench.select_workload(a).choices()) == 64
    for spec, T in (("cartesian:2,3", 9), ("seeded:256", 257), ("cartesian:10,10,10", 1111)):
        a.tree = spec
        wl = bench.select_workload(a)
        assert len(wl.choices()) + 1 == T and wl.name.endswith(spec)
    a.tree = "cartesian:2,2,2,2,2,2"   # deeper than the workload's 5 heads
    try:
        bench.select_workload(a)
        raise AssertionError("a tree deeper than the heads was accepted")
    except SystemExit:
        pass
