"""The multi-rank benchmark path on CPU (gloo, world size 2).

The layer has no exchange step: under torchrun every rank runs an independent replica and
the timing is the maximum over ranks; the reference arm (the float64 oracle) runs on rank 0
alone. These tests launch bench.py the way the two-GPU job is launched, with the gloo
backend on the CPU, and check the rank-level plumbing (no GPU, no data-path collective).
"""
import contextlib
import io
import json
import os
import socket
import subprocess
import sys
import time

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


def _repo_arm_worker(rank, world, port, q):
    """bench.run_ours on this rank with the GPU measurement replaced by a stub that sleeps
    (rank + 1) * 20 ms per step inside bench.timed (barriers, wall timer, max over ranks)."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    seen = {}

    def fake_measure(args, wl, ctx, seed, steps, warmup, **kw):
        seen["seed"], seen["steps"] = seed, steps
        ms = bench.timed(ctx, steps, lambda i: time.sleep(0.02 * (ctx.rank + 1)),
                         lambda: None, bench.WallTimer())
        T, k, H, I = wl.T, wl.k, wl.H, wl.I
        return {"ms": ms, "e2e_ms": 2 * ms, "e2e_serial_ms": 3 * ms, "io_bytes": T * H * 4,
                "stage": {n: ms / 6 for n in ("route", "align", "gather", "gemm1", "gemm2",
                                              "combine")},
                "clocks": {"sm_mhz": None}, "npp": T * k, "active": wl.E,
                "local_rows": T * k, "small": False, "dec": False, "n_copies": 1, "wbytes": 4,
                "launches_per_step": 7, "graph": True, "T": T, "k": k, "E": wl.E, "H": H,
                "I": I, "block_m": 16}

    args = bench.parse(["--gpus", str(world), "--steps", "3", "--warmup", "1",
                        "--workload", "tiny-f32", "--no-cpu-baseline"])
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_ours(args, bench.workload("tiny-f32"), measure=fake_measure)
    q.put((rank, seen["seed"], seen["steps"], buf.getvalue()))


def test_repo_arm_rank_plumbing_gloo():
    """Two ranks: each measures its own replica with its own seed; the step time is the
    slower rank's (max over ranks, taken between barriers); rank 0 alone prints one line
    whose value sums both ranks' useful FLOPs and whose global batch is 2 T."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_repo_arm_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, seed0, steps0, out0), (r1, seed1, steps1, out1) = got
    assert seed1 - seed0 == 1000 and steps0 == steps1 == 3
    assert out1.strip() == ""
    lines = [l for l in out0.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["scaling"] == "weak" and "sweep" not in d
    assert d["ms_per_step"] >= 40.0            # rank 1's 40 ms steps, not rank 0's 20 ms
    sys.path.insert(0, ROOT)
    import moe_inputs as mi
    wl = mi.TINY_F32
    flops = 6 * wl.T * wl.k * wl.H * wl.I
    assert abs(d["value"] - 2 * flops / (d["ms_per_step"] * 1e-3) / 1e12) <= 1e-9 * d["value"]
    assert d["config"]["global_batch"] == 2 * wl.T and d["config"]["parallelism"] == "replicas x2"
    assert abs(d["e2e"]["value"] - d["value"] / 2) <= 1e-9 * d["value"]
    assert abs(d["e2e"]["serial"]["value"] - d["value"] / 3) <= 1e-9 * d["value"]
    assert d["gpu_launches"] == 7 * 3


def test_both_arms_print_the_same_config():
    """The reference arm's config is the repo arm's static config (same keys, same values)."""
    sys.path.insert(0, ROOT)
    import bench
    wl = bench.workload("mixtral-prefill")
    a = bench.static_config(wl, 1)
    assert a["workload"] == "mixtral-prefill" and a["block_m"] == 128 and a["T"] == 4096
    assert set(a) == {"workload", "expert_weights", "T", "H", "I", "E", "k", "n_shared", "mode",
                      "global_batch", "parallelism", "l2", "block_m"}
