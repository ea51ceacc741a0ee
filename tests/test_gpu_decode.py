"""The decode path of moe_forward: batches of at most 8 tokens and 32 routed slots take top-k
and the align table from one small CTA (expert map applied there); and the FP8 prefill path,
which converts each grouped GEMM's weights to bf16 before the GEMM.

Its results must be the separate entry points' bits (same device arithmetic, same summation
orders), its intermediates the same tables, and it must replay from a CUDA graph.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from _helpers import (assert_close, enforce_margins, oracle_logits, oracle_route_from_logits,
                      to_np, weights_for_oracle)
import oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    from routing_grouped_gemm_router_gb300 import _lib
    _lib.moe_device_status(True)
    yield _lib
    torch.cuda.synchronize()
    assert _lib.moe_device_status(True) == 0, "a kernel recorded a device fault"


def _dev(t):
    return None if t is None else t.to(DEV).contiguous()


CASES = [
    ("T1", mi.Workload("dec-T1", T=1, H=1024, I=768, E=32, k=4, dtype="bf16", seed=41), 0, None),
    ("T2-ragged", mi.Workload("dec-T2", T=2, H=1000, I=776, E=16, k=4, dtype="bf16", seed=42),
     0, None),
    ("T2-grouped", mi.Workload("dec-grp", T=2, H=512, I=384, E=64, k=8, dtype="bf16",
                               mode=mi.ROUTE_SIGMOID_GROUPED, scale=2.5, n_group=8,
                               topk_group=4, select_bias_std=0.05, seed=43), 0, None),
    ("T2-shared", mi.Workload("dec-sh", T=2, H=512, I=512, E=16, k=4, dtype="bf16", seed=44),
     1, None),
    ("T2-map-half", mi.Workload("dec-map", T=2, H=512, I=512, E=16, k=4, dtype="bf16", seed=45),
     0, "half"),
    ("T1-E300", mi.Workload("dec-300", T=1, H=256, I=256, E=300, k=6, dtype="bf16", seed=46),
     0, None),
    # FP8 E4M3 expert weights with 128 x 128 block scales: one token, and eight tokens (two
    # passes of four rows where an expert holds more than four)
    ("T1-fp8", mi.Workload("dec-f8", T=1, H=1024, I=768, E=32, k=4, dtype="bf16", seed=50),
     0, "fp8"),
    ("T8-fp8", mi.Workload("dec-f8b", T=8, H=512, I=640, E=8, k=4, dtype="bf16", seed=51),
     0, "fp8"),
    # FP8 weights at prefill: moe_forward turns each GEMM's weights into bf16 in its workspace
    # and runs the bf16 kernels, the separate entry points convert inside the GEMM; the same
    # operands (code times scale, rounded once), so the same bits. Scales that are not powers
    # of two, a shared expert, half of the experts remote (every slot converted then).
    ("T1024-fp8", mi.Workload("pre-f8", T=1024, H=512, I=384, E=8, k=2, dtype="bf16", seed=52),
     0, "fp8"),
    ("T1024-fp8-any", mi.Workload("pre-f8a", T=1024, H=384, I=272, E=8, k=2, dtype="bf16",
                                  seed=53), 0, "fp8-any"),
    ("T1024-fp8-shared", mi.Workload("pre-f8s", T=1024, H=512, I=256, E=8, k=2, dtype="bf16",
                                     seed=54), 1, "fp8"),
    ("T1024-fp8-map", mi.Workload("pre-f8m", T=1024, H=512, I=384, E=8, k=2, dtype="bf16",
                                  seed=55), 0, "fp8-half"),
]


def _setup(L, wl, n_shared, variant):
    inp = mi.make_layer(wl, "cpu")
    enforce_margins(inp)
    W13, W2 = inp.W13, inp.W2
    if n_shared:
        g = torch.Generator().manual_seed(wl.seed + 5)
        W13 = torch.cat([W13, (torch.randn(n_shared, 2 * wl.I, wl.H, generator=g)
                               / wl.H ** 0.5).bfloat16()])
        W2 = torch.cat([W2, (torch.randn(n_shared, wl.H, wl.I, generator=g)
                             / wl.I ** 0.5).bfloat16()])
    Ee = wl.E + n_shared
    emap = None
    scales = {}
    if variant and variant.startswith("fp8"):
        (W13, s13), (W2, s2) = mi.quantize_fp8_w13(W13), mi.quantize_fp8_blocks(W2)
        if variant == "fp8-any":
            g = torch.Generator().manual_seed(wl.seed + 7)
            s13 = s13 * (1.0 + torch.rand(s13.shape, generator=g))
            s2 = s2 * (1.0 + torch.rand(s2.shape, generator=g))
        scales = dict(w13_scale=_dev(s13), w2_scale=_dev(s2))
    if variant in ("half", "fp8-half"):
        emap = torch.tensor([e if e % 2 == 0 else -1 for e in range(Ee)], dtype=torch.int32)
    elif variant == "none":
        emap = torch.full((Ee,), -1, dtype=torch.int32)
    cfg_t = dict(logit_bias=_dev(inp.logit_bias), select_bias=_dev(inp.select_bias),
                 expert_map=_dev(emap), **scales)
    cfg = L.make_config(wl.T, wl.H, wl.I, wl.E, wl.k, L.MOE_BF16, wl.mode, wl.renormalize,
                        wl.scale, wl.n_group, wl.topk_group, cfg_t["logit_bias"],
                        cfg_t["select_bias"], cfg_t["expert_map"], n_shared,
                        scales.get("w13_scale"), scales.get("w2_scale"))
    return inp, _dev(inp.x), _dev(inp.Wg), _dev(W13), _dev(W2), emap, cfg, cfg_t


def _separate(L, wl, cfg, x, Wg, W13, W2, n_shared, emap_d):
    """The layer through the separate entry points (route, align, expert map, GEMMs, combine)."""
    T, kk, Ee, H, I = wl.T, wl.k + n_shared, wl.E + n_shared, wl.H, wl.I
    B = L.moe_block_m(cfg)
    mp = L.moe_max_padded_rows(T, kk, Ee, B)
    r = {"logits": torch.empty(T, wl.E, device=DEV),
         "ids": torch.empty(T, kk, dtype=torch.int32, device=DEV),
         "w": torch.empty(T, kk, device=DEV),
         "sid": torch.empty(mp, dtype=torch.int32, device=DEV),
         "eid": torch.empty(mp // B, dtype=torch.int32, device=DEV),
         "npp": torch.empty(1, dtype=torch.int32, device=DEV),
         "counts": torch.empty(Ee, dtype=torch.int32, device=DEV),
         "act": torch.empty(mp, I, dtype=torch.bfloat16, device=DEV),
         "y": torch.zeros(T * kk, H, dtype=torch.bfloat16, device=DEV),
         "out": torch.empty(T, H, dtype=torch.bfloat16, device=DEV)}
    L.moe_route(cfg, x, Wg, r["logits"], r["ids"], r["w"])
    L.moe_align(r["ids"], T, kk, Ee, B, r["sid"], r["eid"], r["npp"], r["counts"])
    if emap_d is not None:
        L.moe_apply_expert_map(r["eid"], mp // B, emap_d, Ee)
    g1b = L.moe_expert_gemm1_workspace_size(cfg, B)
    g1 = torch.empty(max(g1b, 1), dtype=torch.uint8, device=DEV)
    L.moe_expert_gemm1(cfg, x, W13, r["sid"], r["eid"], r["npp"], B, r["act"], g1, g1b)
    g2b = L.moe_expert_gemm2_workspace_size(cfg, B)
    g2 = torch.empty(max(g2b, 1), dtype=torch.uint8, device=DEV)
    L.moe_expert_gemm2(cfg, r["act"], W2, r["sid"], r["eid"], r["npp"], B, r["w"], r["y"],
                       g2, g2b)
    if emap_d is not None:
        L.moe_combine_local(r["y"], r["ids"], emap_d, Ee, T, kk, H, L.MOE_BF16, r["out"])
    else:
        L.moe_combine(r["y"], T, kk, H, L.MOE_BF16, r["out"])
    return r


@pytest.mark.parametrize("name,wl,n_shared,variant", CASES, ids=[c[0] for c in CASES])
def test_decode_forward_is_the_separate_entry_points_bit_for_bit(L, name, wl, n_shared, variant):
    inp, x, Wg, W13, W2, emap, cfg, keep = _setup(L, wl, n_shared, variant)
    T, kk, H = wl.T, wl.k + n_shared, wl.H
    lay = L.moe_workspace_layout(cfg)
    ws = torch.empty(lay.total, dtype=torch.uint8, device=DEV)
    out = torch.full((T, H), 7.0, dtype=torch.bfloat16, device=DEV)
    L.moe_forward(cfg, x, Wg, W13, W2, out, ws, lay.total)
    ref = _separate(L, wl, cfg, x, Wg, W13, W2, n_shared, keep["expert_map"])
    logits = torch.empty(T, wl.E, device=DEV)
    L.moe_route_logits(cfg, x, Wg, logits)
    torch.cuda.synchronize()
    assert torch.equal(logits, ref["logits"])
    assert torch.equal(out, ref["out"])

    def view(off, count, dtype):
        esz = torch.tensor([], dtype=dtype).element_size()
        return ws[off:off + count * esz].view(dtype)
    n = T * kk
    assert torch.equal(view(lay.topk_ids, n, torch.int32), ref["ids"].flatten())
    assert torch.equal(view(lay.topk_w, n, torch.float32), ref["w"].flatten())
    assert torch.equal(view(lay.sorted_ids, lay.max_padded, torch.int32), ref["sid"])
    assert torch.equal(view(lay.expert_ids, lay.max_padded // lay.block_m, torch.int32),
                       ref["eid"])
    assert torch.equal(view(lay.num_post_padded, 1, torch.int32), ref["npp"])
    assert torch.equal(view(lay.counts, wl.E + n_shared, torch.int32), ref["counts"])
    ids = ref["ids"].flatten().cpu()
    local = torch.ones(n, dtype=torch.bool) if emap is None else emap[ids.long()] >= 0
    y = view(lay.y, n * H, torch.bfloat16).view(n, H)
    assert torch.equal(y[local.to(DEV)], ref["y"][local.to(DEV)])
    # the oracle (both readings of the routing, float64 experts)
    if n_shared == 0:
        sb = to_np(inp.select_bias) if inp.select_bias is not None else None
        oids, ow = oracle_route_from_logits(oracle_logits(inp), wl, sb)
        assert np.array_equal(to_np(ref["ids"]), oids)
        if variant and variant.startswith("fp8"):
            W13o = O.dequant_w13(W13.cpu().numpy(), keep["w13_scale"].double().cpu().numpy())
            W2o = O.dequant_blockwise(W2.cpu().numpy(), keep["w2_scale"].double().cpu().numpy())
        else:
            W13o, W2o = weights_for_oracle(W13.cpu()), weights_for_oracle(W2.cpu())
        refo = O.moe_loop(to_np(inp.x), oids, ow, W13o, W2o,
                          expert_map=None if emap is None else emap.numpy())
        assert_close(to_np(out), refo, "bf16")


def test_decode_all_experts_remote_gives_zero(L):
    wl = mi.Workload("dec-none", T=2, H=256, I=256, E=8, k=2, dtype="bf16", seed=47)
    inp, x, Wg, W13, W2, emap, cfg, keep = _setup(L, wl, 0, "none")
    from routing_grouped_gemm_router_gb300.layer import MoELayer
    layer = MoELayer(Wg, W13, W2, wl.k, expert_map=keep["expert_map"])
    out = layer(x, torch.full((wl.T, wl.H), 3.0, dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    mids = layer.intermediates(wl.T)
    assert torch.all(mids["expert_ids"] == -1)


@pytest.mark.parametrize("T", [1, 2])
def test_decode_graph_capture_and_replay(L, T):
    wl = mi.Workload("dec-graph", T=T, H=2880, I=2880, E=128, k=4, dtype="bf16", seed=48)
    inp = mi.make_layer(wl, DEV)
    from routing_grouped_gemm_router_gb300.layer import MoELayer
    layer = MoELayer(inp.Wg, inp.W13, inp.W2, wl.k)
    x_static = inp.x.clone()
    out_static = torch.empty_like(x_static)
    layer(x_static, out_static)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            layer(x_static, out_static)
    torch.cuda.current_stream().wait_stream(s)
    for seed in (1, 2, 3):
        xn = torch.randn(T, wl.H, generator=torch.Generator().manual_seed(seed)).bfloat16()
        x_static.copy_(xn.to(DEV))
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        eager = layer(x_static.clone())
        torch.cuda.synchronize()
        assert torch.equal(out_static, eager)
