"""The multi-rank benchmark path on CPU (gloo, world size 2).

The layer has no exchange step: under torchrun every rank runs an independent replica and
the timing is the maximum over ranks; the reference arm (the float64 oracle) runs on rank 0
alone. These tests launch bench.py the way the two-GPU job is launched, with the gloo
backend on the CPU, and check the rank-level plumbing (no GPU, no data-path collective).
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist, r, w, local = bench.dist_setup(world)
    m = bench.max_over_ranks(dist, float(10 * (r + 1)), "cpu")
    dist.destroy_process_group()
    q.put((r, w, local, m))


def test_dist_setup_and_max_over_ranks_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 0, 20.0), (1, 2, 1, 20.0)]


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` under torchrun: rank 0 prints one JSON line, rank 1 exits 0
    without work (the oracle runs once, on the host cores)."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--workload", "tiny-f32", "--steps", "2",
           "--warmup", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["config"]["workload"] == "tiny-f32" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
