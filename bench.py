"""Benchmark of the fused MoE layer (one step = route -> align -> GEMM1+SwiGLU -> GEMM2 ->
combine over one batch of T tokens).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line. ``value`` is the layer's useful throughput, 6*T*k*H*I FLOPs per step
(padding and router excluded) over the device-timed step, summed over ranks; ``e2e`` is the
same metric through the public API (MoELayer -> moe_forward) with the tokens copied in from
pinned host memory and the output read back inside the timed region. Under torchrun each
rank runs its own replica of the layer on its own tokens (weak scaling, no data-path
collective); the timing takes the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import moe_inputs as mi  # noqa: E402

METRIC = "MoE layer TFLOPS (6*T*k*H*I/s) & % BF16 peak; decode weight GB/s vs HBM"
DEFAULT_WORKLOAD = "mixtral-prefill"


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD,
                   help="mixtral-prefill | qwen3-skewed | deepseek-v3 | gpt-oss-decode@T=<n>")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample-tokens", type=int, default=0)
    p.add_argument("--no-graph", action="store_true",
                   help="time eager launches instead of CUDA-graph replays of the step")
    p.add_argument("--shared", type=int, default=0,
                   help="shared experts (weight 1 on every token) added to the routed ones")
    p.add_argument("--masked", action="store_true",
                   help="fixed-capacity expert layout (tokens already bucketed per expert, no "
                        "router/align): moe_masked_forward on the workload's shape")
    p.add_argument("--ep-half", action="store_true",
                   help="expert parallelism: odd experts on another device (expert_map -1); "
                        "the metric counts the rows of local experts only")
    p.add_argument("--fp8", action="store_true",
                   help="FP8 E4M3 expert weights with 128x128 block scales (the seeded bf16 "
                        "weights quantised); tokens, router and GEMM arithmetic stay bf16")
    p.add_argument("--tokens", type=int, default=0,
                   help="override T of the workload (smaller cases for profiling)")
    p.add_argument("--experts", type=int, default=0,
                   help="override E of the workload (smaller cases for profiling)")
    p.add_argument("--inter", type=int, default=0,
                   help="override I of the workload (captures of the routing kernels, which "
                        "depend on T, H, E and k only, with small expert weights)")
    p.add_argument("--no-sweep", action="store_true",
                   help="only the headline workload (the default run also measures the other "
                        "prefill shapes, the decode sweep and FP8 decode)")
    p.add_argument("--sweep-steps", type=int, default=10)
    return p.parse_args(argv)


def workload(name: str) -> mi.Workload:
    if name.startswith("gpt-oss-decode@T="):
        return mi.GPTOSS.with_T(int(name.split("=")[1]))
    return mi.WORKLOADS[name]


def is_decode(wl):
    return wl.name.startswith("gpt-oss-decode")


def peaks():
    """(HBM GB/s, bf16 burst TF/s, bf16 sustained TF/s, source)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# Headers left out of a kernel's source hash: common.cuh is the library's internal launch
# table (host declarations of every launcher) plus one-line helpers, included everywhere; an
# entry point added there does not change any kernel.
HASH_SKIP = ("common.cuh",)


def source_hash(src_path: str) -> str:
    """sha256 of a kernel's source: the file, then every header it includes from its own
    directory (recursively, each once, in include order; HASH_SKIP excepted), so that an edit
    to a kernel body kept in a header voids the summaries taken on the old code."""
    d, seen = os.path.dirname(src_path), []

    def visit(path):
        if path in seen:
            return
        seen.append(path)
        for m in re.finditer(r'#include "([^"]+)"', open(path).read()):
            q = os.path.join(d, m.group(1))
            if os.path.exists(q) and m.group(1) not in HASH_SKIP:
                visit(q)
    visit(src_path)
    h = hashlib.sha256()
    for path in seen:
        h.update(open(path, "rb").read())
    return h.hexdigest()


def profile_traffic(kernel: str, wl_name: str, active: int, src_path: str):
    """DRAM bytes per launch recorded in a committed ncu summary, if the kernel source it
    was taken on is unchanged (the summary stores the source's sha256); else None.

    A summary holds either a per-launch figure of its own workload, or a figure per active
    expert taken on a smaller expert count of the same launch shape (the same rows per
    expert, the same split), scaled here by the launch's active experts; the workloads it
    stands for are listed on its traffic_workloads line (names without the @E= suffix)."""
    base = wl_name.split("@")[0]
    path = os.path.join(ROOT, "profiles", f"{kernel}_{base}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", txt)
    if not h or source_hash(src_path) != h.group(1):
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if m:
        return float(m.group(1)) if wl_name == base else None
    m = re.search(r"traffic_bytes_per_active_expert:\s*([0-9.eE+]+)", txt)
    w = re.search(r"traffic_workloads:(.*)", txt)
    name = re.sub(r"@E=\d+", "", wl_name)
    if m and w and name in w.group(1).split():
        return float(m.group(1)) * active
    return None


class ClockSampler:
    """nvidia-smi sampled every 100 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    import torch
    if n_gpus > 1 or int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist, dist.get_rank(), dist.get_world_size(), local
    return None, 0, 1, 0


def max_over_ranks(dist, v: float, device) -> float:
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------ CPU oracle

def time_oracle(wl, x, Wg, W13, W2, lb, sb, n_tokens):
    """The float64 oracle (route + per-expert loop), as it stands, on the first ``n_tokens``
    tokens of the same layer. Returns (seconds, tokens, threads)."""
    import numpy as np
    import oracle as O
    xs = x[:n_tokens]
    t0 = time.perf_counter()
    logits = O.router_logits(xs, Wg, lb if wl.mode == 0 else None)
    ids, w = O.route(logits, wl.k, wl.mode, wl.renormalize, wl.scale, wl.n_group,
                     wl.topk_group, sb)
    out = O.moe_loop(xs, ids, w, W13, W2)
    dt = time.perf_counter() - t0
    assert np.isfinite(out).all()
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return dt, xs.shape[0], threads


def host_copies(inp):
    """Host copies for the oracle: fp64 tokens/router, raw bf16 bits of the expert weights."""
    import numpy as np
    import torch

    def bits(t):
        if t.dtype != torch.bfloat16:
            return t.detach().double().cpu().numpy()
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    def f64(t):
        return t.detach().float().cpu().double().numpy()
    lb = f64(inp.logit_bias) if inp.logit_bias is not None else None
    sb = f64(inp.select_bias) if inp.select_bias is not None else None
    return f64(inp.x), f64(inp.Wg), bits(inp.W13), bits(inp.W2), lb, sb


def default_sample(wl):
    """Tokens per oracle pass: about 10-20 s of float64 work on a 16-core host."""
    return {"mixtral-prefill": 1536, "qwen3-skewed": 768,
            "deepseek-v3": 256}.get(wl.name.split("@")[0], wl.T)


# ------------------------------------------------------------------------------ ranks

class RankCtx:
    """This process's place in the job: one replica of the layer per rank (no data-path
    collective); the process group only serves the barriers around timed regions and the
    max-over-ranks of the timings."""

    def __init__(self, dist, rank, world, local):
        self.dist, self.rank, self.world, self.local = dist, rank, world, local

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, v, device="cpu"):
        return max_over_ranks(self.dist, v, device)

    def finish(self):
        if self.dist is not None:
            self.dist.barrier()
            self.dist.destroy_process_group()


class CudaTimer:
    """Device time between two CUDA events recorded on the launching stream."""

    def __init__(self, stream):
        import torch
        self.stream = stream
        self.e0 = torch.cuda.Event(enable_timing=True)
        self.e1 = torch.cuda.Event(enable_timing=True)

    def start(self):
        self.e0.record(self.stream)

    def stop(self):
        self.e1.record(self.stream)

    def ms(self):
        return self.e0.elapsed_time(self.e1)


class WallTimer:
    """Host wall time (the CPU-only plumbing tests)."""

    def start(self):
        self.t0 = time.perf_counter()

    def stop(self):
        self.t1 = time.perf_counter()

    def ms(self):
        return (self.t1 - self.t0) * 1e3


def timed(ctx, steps, run, sync, timer, device="cpu"):
    """Time `steps` calls of run(i): barrier and sync before, timer around the loop, sync and
    barrier after; returns ms per step, the maximum over ranks."""
    ctx.barrier()
    sync()
    timer.start()
    for i in range(steps):
        run(i)
    timer.stop()
    sync()
    ctx.barrier()
    return ctx.max(timer.ms() / steps, device)


def workload_label(wl, shared=0, fp8=False, ep_half=False):
    return (wl.name + ("+ep-half" if ep_half else "") + (f"+shared{shared}" if shared else "")
            + ("+fp8" if fp8 else ""))


def static_config(wl, world, shared=0, fp8=False, ep_half=False):
    """The `config` of a bench line: the workload and how it is laid out and timed. Both arms
    print exactly this (nothing measured goes in here)."""
    wbytes = 1 if fp8 else (2 if wl.dtype == "bf16" else 4)
    E = wl.E + shared
    if is_decode(wl):
        l2 = ("3 copies of the expert weights rotated between steps, so each step streams its "
              "active experts from HBM (L2 126 MB)")
    else:
        l2 = f"inputs larger than L2 (expert weights {E * 3 * wl.H * wl.I * wbytes / 1e9:.2f} GB)"
    return {"workload": workload_label(wl, shared, fp8, ep_half),
            "expert_weights": "fp8-e4m3, fp32 scale per 128x128 block" if fp8 else
                              ("bf16" if wl.dtype == "bf16" else "f32"),
            "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k, "n_shared": shared,
            "mode": "sigmoid-grouped" if wl.mode else "softmax",
            "global_batch": wl.T * world, "parallelism": f"replicas x{world}", "l2": l2,
            "block_m": 128 if wl.dtype == "bf16" else 16}


# ------------------------------------------------------------------------------ arms

def run_reference(args, wl):
    """Reference arm: the float64 CPU oracle on the host cores, rank 0 only."""
    import torch
    dist, rank, world, local = dist_setup(args.gpus)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = mi.make_layer(wl, dev, seed=wl.seed)
    x, Wg, W13, W2, lb, sb = host_copies(inp)
    del inp
    n = args.cpu_sample_tokens or default_sample(wl)
    for _ in range(max(0, args.warmup)):
        time_oracle(wl, x, Wg, W13, W2, lb, sb, min(n, 2))
    secs, threads = 0.0, 1
    for _ in range(args.steps):
        dt, n, threads = time_oracle(wl, x, Wg, W13, W2, lb, sb, n)
        secs += dt
    flops = 6 * n * wl.k * wl.H * wl.I
    val = flops * args.steps / secs / 1e12
    line = {"metric": METRIC, "value": val, "unit": "TFLOPS", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": static_config(wl, args.gpus),
            "cpu_baseline": {"value": val, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                             "sample": f"first {n} of {wl.T} tokens per step, float64 oracle "
                                       "(router + per-expert loop)"},
            "e2e": {"value": val, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def measure_layer(args, wl, ctx, seed, steps, warmup, shared=0, fp8=False, ep_half=False,
                  e2e=True, cpu_baseline=False):
    """One layer configuration on this rank's GPU: CUDA-graph replays of moe_forward (the
    device-timed steps), the same stages launched eagerly with events between them, and
    (e2e) the public API with host copies of the tokens and the output. Times are maxima
    over ranks. Returns a dict of raw measurements (summarize() turns it into line fields)."""
    import torch
    dev = torch.device("cuda", ctx.local)
    torch.cuda.set_device(dev)
    from routing_grouped_gemm_router_gb300 import _lib as L  # fails loudly if not built
    from routing_grouped_gemm_router_gb300.layer import MoELayer

    inp = mi.make_layer(wl, dev, seed=seed)
    if shared:  # shared experts' weights follow the routed experts'
        g = torch.Generator(device=dev)
        g.manual_seed(wl.seed + 77)
        inp.W13 = torch.cat([inp.W13, (torch.randn(shared, 2 * wl.I, wl.H, generator=g,
                                                   device=dev) / wl.H ** 0.5).to(inp.W13.dtype)])
        inp.W2 = torch.cat([inp.W2, (torch.randn(shared, wl.H, wl.I, generator=g,
                                                 device=dev) / wl.I ** 0.5).to(inp.W2.dtype)])
    sc13 = sc2 = None
    if fp8:  # codes + block scales replace the bf16 expert weights
        inp.W13, sc13 = mi.quantize_fp8_w13(inp.W13)
        inp.W2, sc2 = mi.quantize_fp8_blocks(inp.W2)
        torch.cuda.empty_cache()
    emap = None
    if ep_half:
        emap = torch.tensor([e if e % 2 == 0 else -1 for e in range(wl.E + shared)],
                            dtype=torch.int32, device=dev)
    # Decode streams only the active experts' weights (gpt-oss T=1: 0.2 GB, not much more
    # than the 126 MB L2): successive steps rotate over three copies of the expert weights so
    # that each step reads them from HBM, not from L2 left warm by the step before.
    n_copies = 3 if is_decode(wl) else 1
    W13s = [inp.W13] + [inp.W13.clone() for _ in range(n_copies - 1)]
    W2s = [inp.W2] + [inp.W2.clone() for _ in range(n_copies - 1)]
    layers = [MoELayer(inp.Wg, W13s[c], W2s[c], wl.k, wl.mode, wl.renormalize, wl.scale,
                       wl.n_group, wl.topk_group, inp.logit_bias, inp.select_bias, emap,
                       n_shared=shared, w13_scale=sc13, w2_scale=sc2)
              for c in range(n_copies)]
    layer = layers[0]
    wbytes = 1 if fp8 else inp.x.element_size()  # bytes per expert weight
    # the align step, the grouped GEMMs and the combine see shared experts as ordinary ones
    T, k, E, H, I = wl.T, wl.k + shared, wl.E + shared, wl.H, wl.I
    cfg = layer.config(T)
    ws, lay = layer.workspace(T)
    B = lay.block_m
    base = ws.data_ptr()
    p = {n: base + getattr(lay, n) for n in ("logits", "topk_ids", "topk_w", "sorted_ids",
                                               "expert_ids", "num_post_padded", "counts",
                                               "align_scratch", "act", "xs", "y", "gemm_scratch")}
    ws_gemm = lay.total - lay.gemm_scratch
    ws_align = lay.act - lay.align_scratch
    ws_xs = lay.y - lay.xs
    out = torch.empty(T, H, dtype=inp.x.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    # bf16 GEMM1 = row gather + tensor-core GEMM, timed apart; the library says which grouped
    # GEMM kernels the batch runs: small batches the CUDA-core kernels (which read the token
    # rows in place), other decode batches the decode tensor-core kernel
    kind = L.moe_gemm_kernel(cfg)
    small = kind == L.MOE_GEMM_SMALL_BATCH
    dec = kind == L.MOE_GEMM_DECODE_TC
    gathered = wl.dtype == "bf16" and not small
    # FP8 weights at prefill: moe_forward writes each GEMM's weights as bf16 into the
    # workspace's GEMM scratch and runs the bf16 kernels on them (the region is empty otherwise)
    dq = fp8 and lay.total > lay.gemm_scratch
    cfg_dq = layer.config(T)
    if dq:
        cfg_dq.weight_format, cfg_dq.w13_scale, cfg_dq.w2_scale = L.MOE_WEIGHTS_NATIVE, None, None
    dq_counts = None if emap is not None else p["counts"]

    def step(ev=None, sh=sh, c=0):
        # The same kernels moe_forward enqueues, called stage by stage so that CUDA events
        # between them give each stage's device time.
        if ev is not None:
            ev[0].record(stream)
        L.moe_route(cfg, inp.x, inp.Wg, p["logits"], p["topk_ids"], p["topk_w"], sh)
        if ev is not None:
            ev[1].record(stream)
        L.moe_align(p["topk_ids"], T, k, E, B, p["sorted_ids"], p["expert_ids"],
                    p["num_post_padded"], p["counts"], p["align_scratch"], ws_align, sh)
        if emap is not None:
            L.moe_apply_expert_map(p["expert_ids"], lay.max_padded // B, emap, E, sh)
        if ev is not None:
            ev[2].record(stream)
        if gathered:
            L.moe_gather_rows(inp.x, p["sorted_ids"], p["num_post_padded"], T, k, H, cfg.dtype,
                              p["xs"], sh)
        if ev is not None:
            ev[3].record(stream)
        if dq:
            L.moe_dequant_fp8_weights(cfg, 1, W13s[c], dq_counts, p["gemm_scratch"], sh)
        if ev is not None:
            ev[4].record(stream)
        if dq:
            L.moe_expert_gemm1_gathered(cfg_dq, p["xs"], p["gemm_scratch"], p["sorted_ids"],
                                        p["expert_ids"], p["num_post_padded"], B, p["act"],
                                        None, 0, sh)
        elif gathered:
            L.moe_expert_gemm1_gathered(cfg, p["xs"], W13s[c], p["sorted_ids"], p["expert_ids"],
                                        p["num_post_padded"], B, p["act"], p["gemm_scratch"],
                                        ws_gemm, sh)
        else:
            L.moe_expert_gemm1(cfg, inp.x, W13s[c], p["sorted_ids"], p["expert_ids"],
                               p["num_post_padded"], B, p["act"], p["xs"], ws_xs, sh)
        if ev is not None:
            ev[5].record(stream)
        if dq:
            L.moe_dequant_fp8_weights(cfg, 2, W2s[c], dq_counts, p["gemm_scratch"], sh)
        if ev is not None:
            ev[6].record(stream)
        if dq:
            L.moe_expert_gemm2(cfg_dq, p["act"], p["gemm_scratch"], p["sorted_ids"],
                               p["expert_ids"], p["num_post_padded"], B, p["topk_w"], p["y"],
                               None, 0, sh)
        else:
            L.moe_expert_gemm2(cfg, p["act"], W2s[c], p["sorted_ids"], p["expert_ids"],
                               p["num_post_padded"], B, p["topk_w"], p["y"], p["gemm_scratch"],
                               ws_gemm, sh)
        if ev is not None:
            ev[7].record(stream)
        if emap is not None:
            L.moe_combine_local(p["y"], p["topk_ids"], emap, E, T, k, H, cfg.dtype, out, sh)
        else:
            L.moe_combine(p["y"], T, k, H, cfg.dtype, out, sh)
        if ev is not None:
            ev[8].record(stream)

    def forward(sh=sh, c=0):
        # the timed step: the public entry point, moe_forward, with the workspace above
        L.moe_forward(cfg, inp.x, inp.Wg, W13s[c], W2s[c], out, ws, lay.total, sh)

    # kernels moe_forward enqueues: router GEMM + top-k, align (one kernel up to 4096 rows,
    # else three; up to 8 tokens top-k and align are one kernel), expert map (applied by the
    # routing kernel of batches of at most 32 slots), row gather (bf16 tensor-core path),
    # GEMM1, GEMM2 and the combine
    tiny = T <= 8 and T * k <= 32
    routing_launches = 2 if (T <= 8 and T * k <= 4096) else 2 + (1 if T * k <= 4096 else 3)
    if tiny and T == 1 and wl.dtype == "bf16":
        routing_launches = 1  # one token: router, top-k and table in one cluster launch
    launches_per_step = routing_launches + (1 if (emap is not None and not tiny) else 0) + \
        (1 if gathered else 0) + 3 + (2 if dq else 0)

    for _ in range(max(3, warmup)):
        step()
        forward()
    torch.cuda.synchronize()
    npp = int(ws[lay.num_post_padded:lay.num_post_padded + 4].view(torch.int32).item())
    counts = ws[lay.counts:lay.counts + 4 * E].view(torch.int32).cpu()
    if emap is not None:  # only the local experts' rows and weights are this device's work
        counts = counts * (emap.cpu() >= 0)
    active = int((counts > 0).sum())
    local_rows = int(counts.sum())

    # ---- the step captured once in a CUDA graph (no host work or launch gaps in the timing)
    graphs = []
    if not args.no_graph:
        for c in range(n_copies):
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cap):
                with torch.cuda.graph(g, stream=cap):
                    forward(sh=cap.cuda_stream, c=c)
            stream.wait_stream(cap)
            graphs.append(g)
        for _ in range(3):
            for g in graphs:
                g.replay()
        torch.cuda.synchronize()

    def run_step(i):
        if graphs:
            graphs[i % n_copies].replay()
        else:
            forward(c=i % n_copies)

    # ---- device-timed steps (inputs resident in HBM; expert weights larger than L2)
    sampler = ClockSampler(ctx.local)
    sampler.start()
    time.sleep(0.3)
    ms = timed(ctx, steps, run_step, torch.cuda.synchronize, CudaTimer(stream), dev)
    # per-stage device times: the same steps launched eagerly with CUDA events between stages
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(9)] for _ in range(steps)]
    for i in range(steps):
        step(evs[i], c=i % n_copies)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    stage = {n: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
             for i, n in enumerate(("route", "align", "gather", "dequant1", "gemm1", "dequant2",
                                    "gemm2", "combine"))}
    if not dq:
        del stage["dequant1"], stage["dequant2"]
    res = {"ms": ms, "stage": stage, "clocks": clocks, "npp": npp, "active": active,
           "local_rows": local_rows, "small": bool(small), "dec": bool(dec), "dq": bool(dq),
           "n_copies": n_copies,
           "wbytes": wbytes, "launches_per_step": launches_per_step, "graph": bool(graphs),
           "T": T, "k": k, "E": E, "H": H, "I": I, "block_m": B}
    del graphs

    # ---- end to end through the public API: H2D of x, moe_forward, D2H of out, every step
    if e2e:
        x_host = inp.x.cpu().pin_memory()
        out_host = [torch.empty(T, H, dtype=inp.x.dtype).pin_memory() for _ in range(2)]
        x_dev = [torch.empty_like(inp.x) for _ in range(2)]
        out_dev = [torch.empty_like(out) for _ in range(2)]

        def e2e_serial(i):
            # one stream: the step's input copy, the layer, the output copy, in turn
            x_dev[0].copy_(x_host, non_blocking=True)
            layers[i % n_copies](x_dev[0], out_dev[0])
            out_host[0].copy_(out_dev[0], non_blocking=True)

        # the serving form: input copies and output copies run on two streams of their own
        # with double-buffered device tensors, so step i+1's input copy and step i-1's readback
        # overlap step i's layer. x_dev[j] is refilled after the layer that read it (step i-2)
        # finished, out_dev[j] is rewritten after its readback finished; the copy streams start
        # after the timer's start event and are joined before its stop event, so every step's
        # two copies lie inside the timed region
        cs_in, cs_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]

        def make_overlapped(n_steps):
            def run(i):
                j = i % 2
                if i == 0:
                    cs_in.wait_stream(stream)
                    cs_out.wait_stream(stream)
                if i >= 2:
                    cs_in.wait_event(ev_out[j])     # the layer of step i-2 read x_dev[j]
                with torch.cuda.stream(cs_in):
                    x_dev[j].copy_(x_host, non_blocking=True)
                    ev_in[j].record(cs_in)
                stream.wait_event(ev_in[j])
                if i >= 2:
                    stream.wait_event(ev_done[j])   # step i-2's output has been read back
                layers[i % n_copies](x_dev[j], out_dev[j])
                ev_out[j].record(stream)
                cs_out.wait_event(ev_out[j])
                with torch.cuda.stream(cs_out):
                    out_host[j].copy_(out_dev[j], non_blocking=True)
                    ev_done[j].record(cs_out)
                if i == n_steps - 1:
                    stream.wait_stream(cs_in)
                    stream.wait_stream(cs_out)
            return run

        for i in range(3):
            e2e_serial(i)
        warm = make_overlapped(3)
        for i in range(3):
            warm(i)
        torch.cuda.synchronize()
        res["e2e_serial_ms"] = timed(ctx, steps, e2e_serial, torch.cuda.synchronize,
                                     CudaTimer(stream), dev)
        res["e2e_ms"] = timed(ctx, steps, make_overlapped(steps), torch.cuda.synchronize,
                              CudaTimer(stream), dev)
        res["io_bytes"] = T * H * inp.x.element_size()

    if cpu_baseline:
        del layer, layers, W13s, W2s
        x, Wg, W13, W2, lb, sb = host_copies(inp)
        n = args.cpu_sample_tokens or default_sample(wl)
        dt, n, threads = time_oracle(wl, x, Wg, W13, W2, lb, sb, n)
        res["cpu_baseline"] = {"value": 6 * n * k * H * I / dt / 1e12, "unit": "TFLOPS",
                               "cores": threads, "kind": "oracle",
                               "sample": f"first {n} of {T} tokens, one pass of the float64 "
                                         f"oracle (router + per-expert loop), {dt:.1f} s"}
    return res


def summarize(wl, m, world, fp8=False):
    """Line fields of one measured configuration: the metric (useful TFLOPS, summed over
    ranks), active-expert weight GB/s for weight-bound layers, and the roofline of GEMM1,
    the dominant kernel, against the measured peaks."""
    H, I = m["H"], m["I"]
    flops = 6 * m["local_rows"] * H * I  # useful rows (all T*k rows unless experts are remote)
    value = flops * world / (m["ms"] * 1e-3) / 1e12
    hbm, bf16_burst, bf16_sus, peak_src = peaks()
    wbytes, active = m["wbytes"], m["active"]
    # The bound follows the layer's intensity, useful FLOPs per byte of active expert weights
    # (T*k/A for bf16), against the ridge of the measured peaks: decode and the
    # DeepSeek-V3-shaped layer (128 FLOP/B) stream weights; Mixtral and Qwen3 are compute.
    intensity = flops / max(1, active * 3 * H * I * wbytes)
    hbm_bound = is_decode(wl) or intensity < bf16_burst * 1e12 / (hbm * 1e9)
    # The dominant kernel is timed alone (eager, CUDA events around it): the burst peaks are
    # its denominators.
    g1_ms = m["stage"]["gemm1"]
    if hbm_bound:
        w_bytes = active * 2 * H * I * wbytes   # gate/up weights of every active expert
        roof = {"bound": "hbm", "achieved": w_bytes / (g1_ms * 1e-3) / 1e9, "peak": hbm,
                "unit": "GB/s",
                "kernel": "gemm1 (gate/up grouped GEMV, small batch)" if m["small"] else
                          "gemm1 (gate/up decode grouped GEMM, weights as the 128-row operand)"
                          if m["dec"] else "gemm1 (gate/up grouped GEMM)",
                "algorithmic_bytes_per_launch": w_bytes,
                "peak_kind": f"{peak_src} HBM copy bandwidth"}
    else:
        g1_flops = 4 * m["local_rows"] * H * I
        roof = {"bound": "tensor", "achieved": g1_flops / (g1_ms * 1e-3) / 1e12,
                "peak": bf16_burst, "unit": "TFLOP/s",
                "kernel": "gemm1 (gate/up grouped GEMM + SwiGLU)",
                "algorithmic_flops_per_launch": g1_flops,
                "peak_kind": f"{peak_src} bf16 burst (GEMM1 timed alone, CUDA events)"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    kern, src = (("gemv1", "gemv.cu") if m["small"] else ("gemmdec1", "gemm_dec.cu")
                 if m["dec"] else ("gemm1", "gemm_tc2.cu"))
    src = os.path.join(ROOT, "routing_grouped_gemm_router_gb300", "csrc", src)
    if m.get("dq"):  # FP8 weights at prefill: GEMM1 is the bf16 kernel on bf16 copies
        roof["kernel"] += ", bf16 weights written from the FP8 codes just before"
    roof["traffic"] = profile_traffic(kern + ("_fp8" if fp8 and not m.get("dq") else ""),
                                      wl.name, active, src)
    return _line_fields(wl, m, world, value, intensity, hbm_bound, roof, hbm, bf16_burst)


def _line_fields(wl, m, world, value, intensity, hbm_bound, roof, hbm, bf16_burst):
    H, I, wbytes, active = m["H"], m["I"], m["wbytes"], m["active"]
    f = {"value": value, "ms_per_step": m["ms"], "roofline": roof,
         "intensity_flop_per_weight_byte": intensity,
         "routing": {"num_post_padded": m["npp"], "active_experts": active,
                     "rows": m["local_rows"]}}
    if hbm_bound:
        f["weight_gbs"] = active * 3 * H * I * wbytes * world / (m["ms"] * 1e-3) / 1e9
        f["weight_gbs_frac_of_hbm"] = f["weight_gbs"] / (hbm * world)
    if not is_decode(wl):
        f["frac_of_bf16_peak"] = value / (bf16_burst * world)
        f["frac_of_bf16_peak_kind"] = "layer TFLOPS / measured bf16 burst (CUDA-graph replays)"
    return f


# The rest of the metric, measured in the default run next to the headline (one GPU): the
# other prefill shapes, the decode sweep, FP8 expert weights at decode and at prefill.
SWEEP = [("qwen3-skewed", False), ("deepseek-v3", False),
         ("gpt-oss-decode@T=1", False), ("gpt-oss-decode@T=8", False),
         ("gpt-oss-decode@T=32", False), ("gpt-oss-decode@T=128", False),
         ("gpt-oss-decode@T=1", True), ("gpt-oss-decode@T=8", True),
         ("gpt-oss-decode@T=32", True), ("gpt-oss-decode@T=128", True),
         ("mixtral-prefill", True)]


def run_sweep(args, ctx):
    import torch
    out = []
    for name, fp8 in SWEEP:
        wl = workload(name)
        m = measure_layer(args, wl, ctx, seed=wl.seed, steps=args.sweep_steps,
                          warmup=3, fp8=fp8, e2e=False)
        f = summarize(wl, m, 1, fp8)
        r = f["roofline"]
        entry = {"workload": workload_label(wl, fp8=fp8), "ms": round(m["ms"], 5),
                 "tflops": round(f["value"], 2), "steps": args.sweep_steps,
                 "gemm1_roofline": {k: (round(v, 4) if isinstance(v, float) else v)
                                    for k, v in r.items()},
                 "stages_ms": {n: round(v, 5) for n, v in m["stage"].items()},
                 "routing": f["routing"], "clocks": m["clocks"]}
        for key in ("weight_gbs", "weight_gbs_frac_of_hbm", "frac_of_bf16_peak"):
            if key in f:
                entry[key] = round(f[key], 4)
        out.append(entry)
        del m
        torch.cuda.empty_cache()
    return out


def run_ours(args, wl, measure=None):
    """The repo arm: each rank measures its own replica (seed offset by rank) and rank 0
    prints one line whose value sums the ranks' useful FLOPs over the slowest rank's time."""
    dist, rank, world, local = dist_setup(args.gpus)
    ctx = RankCtx(dist, rank, world, local)
    measure = measure or measure_layer
    headline = rank == 0 and world == 1 and not args.no_cpu_baseline and not args.fp8
    m = measure(args, wl, ctx, seed=wl.seed + 1000 * rank, steps=args.steps,
                warmup=args.warmup, shared=args.shared, fp8=args.fp8, ep_half=args.ep_half,
                e2e=True, cpu_baseline=headline)
    f = summarize(wl, m, world, args.fp8)
    line = {"metric": METRIC, "value": f["value"], "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms"],
            "timing": ("CUDA-graph replays of moe_forward" if m["graph"] else
                       "eager moe_forward calls") + "; stages_ms: the separate entry points, eager",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if wl.dtype == "bf16" else "f32",
            "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights, random init)",
            "config": static_config(wl, world, args.shared, args.fp8, args.ep_half),
            "stages_ms": {n: round(v, 5) for n, v in m["stage"].items()},
            "roofline": f["roofline"],
            "e2e": {"value": f["value"] * m["ms"] / m["e2e_ms"], "unit": "TFLOPS",
                    "h2d_bytes_per_step": m["io_bytes"], "d2h_bytes_per_step": m["io_bytes"],
                    "ms_per_step": m["e2e_ms"],
                    "copies": "every step copies its tokens from pinned host memory and reads "
                              "its output back; the copies run on streams of their own, "
                              "overlapping the neighbouring steps' layers (double-buffered)",
                    "serial": {"value": f["value"] * m["ms"] / m["e2e_serial_ms"],
                               "ms_per_step": m["e2e_serial_ms"],
                               "copies": "input copy, layer, output copy in turn on one stream"}},
            "gpu_launches": m["launches_per_step"] * args.steps,
            "clocks": m["clocks"]}
    for key in ("intensity_flop_per_weight_byte", "routing", "weight_gbs",
                "weight_gbs_frac_of_hbm", "frac_of_bf16_peak", "frac_of_bf16_peak_kind"):
        if key in f:
            line[key] = f[key]
    if "cpu_baseline" in m:
        line["cpu_baseline"] = m["cpu_baseline"]
    if world == 1 and not args.no_sweep and args.workload == DEFAULT_WORKLOAD and \
            not (args.tokens or args.experts or args.inter or args.fp8 or args.shared or
                 args.ep_half):
        line["sweep"] = run_sweep(args, ctx)
    if rank == 0:
        print(json.dumps(line), flush=True)
    ctx.finish()


def run_masked(args, wl):
    """moe_masked_forward on buckets filled by a seeded uniform top-k draw of T tokens."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from routing_grouped_gemm_router_gb300 import _lib as L
    g = torch.Generator(device=dev)
    g.manual_seed(wl.seed)
    T, k, E, H, I = wl.T, wl.k, wl.E, wl.H, wl.I
    ids = torch.rand(T, E, generator=g, device=dev).topk(k, dim=1).indices
    counts = torch.bincount(ids.flatten(), minlength=E).to(torch.int32)
    B = 128
    cap = max(B, (int(counts.max()) + B - 1) // B * B)
    inp = mi.make_layer(wl, dev, seed=wl.seed)
    xm = torch.randn(E, cap, H, generator=g, device=dev).to(torch.bfloat16)
    rw = torch.rand(E, cap, generator=g, device=dev)
    y = torch.empty(E, cap, H, dtype=torch.bfloat16, device=dev)
    cfg = L.make_config(1, H, I, E, 1, L.MOE_BF16)
    wsb = L.moe_masked_workspace_size(cfg, cap)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)

    # three copies of the expert weights rotated between steps (each step reads from HBM)
    W13s = [inp.W13, inp.W13.clone(), inp.W13.clone()]
    W2s = [inp.W2, inp.W2.clone(), inp.W2.clone()]

    def step(sh=None, c=0):
        L.moe_masked_forward(cfg, xm, counts, cap, rw, W13s[c], W2s[c], y, ws, wsb, sh)

    for i in range(max(3, args.warmup)):
        step(c=i % 3)
    graphs = []
    for c in range(3):
        cap_s = torch.cuda.Stream(dev)
        cap_s.wait_stream(torch.cuda.current_stream(dev))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap_s):
            with torch.cuda.graph(g, stream=cap_s):
                step(cap_s.cuda_stream, c)
        torch.cuda.current_stream(dev).wait_stream(cap_s)
        graphs.append(g)
    for _ in range(3):
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        graphs[i % 3].replay()
    e1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    rows = int(counts.sum())
    active = int((counts > 0).sum())
    hbm, _, _, _ = peaks()
    gbs = active * 3 * H * I * 2 / (ms * 1e-3) / 1e9
    line = {"metric": METRIC, "value": 6 * rows * H * I / (ms * 1e-3) / 1e12, "unit": "TFLOPS",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "timing": "CUDA-graph replays of moe_masked_forward",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (uniform top-k draw bucketed per expert)",
            "config": {"workload": wl.name + "+masked", "T": T, "H": H, "I": I, "E": E, "k": k,
                       "capacity": cap, "rows": rows, "active_experts": active,
                       "l2": "3 copies of the expert weights rotated between steps"},
            "weight_gbs": gbs, "weight_gbs_frac_of_hbm": gbs / hbm, "clocks": clocks}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    wl = workload(args.workload)
    if args.tokens:
        wl = wl.with_T(args.tokens)
    if args.experts:
        import dataclasses
        wl = dataclasses.replace(wl, E=args.experts, name=f"{wl.name}@E={args.experts}")
    if args.inter:
        import dataclasses
        wl = dataclasses.replace(wl, I=args.inter, name=f"{wl.name}@I={args.inter}")
    if args.impl == "reference":
        run_reference(args, wl)
    elif args.masked:
        run_masked(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
