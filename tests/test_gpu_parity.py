"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Integer work (ids, counts, sorted_ids, expert_ids, padded total) must be bit-exact;
floating point within the tolerances of tests/_helpers.py. Routing decisions are compared
both ways: the oracle's top-k fed with the GPU's fp32 logits, and the oracle's own float64
routing on inputs whose selection margins exceed 1e-4.
"""
import zlib

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle as O
from oracle import moe_oracle as OM
from _helpers import (TOPK_W_RTOL, assert_close, enforce_margins, oracle_logits,
                      oracle_route_from_logits, to_np, weights_for_oracle)

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


def _layer(L, inp):
    from routing_grouped_gemm_router_gb300.layer import MoELayer
    wl = inp.wl
    return MoELayer(inp.Wg, inp.W13, inp.W2, wl.k, wl.mode, wl.renormalize, wl.scale,
                    wl.n_group, wl.topk_group, inp.logit_bias, inp.select_bias)


def _to_dev(inp):
    f = lambda t: None if t is None else t.to(DEV).contiguous()  # noqa: E731
    return mi.LayerInputs(inp.wl, f(inp.x), f(inp.Wg), f(inp.W13), f(inp.W2), f(inp.logit_bias),
                          f(inp.select_bias))


def _check_routing_and_align(inp, mids):
    """ids/weights/align of one forward against the oracle. Returns the oracle's (ids, w)."""
    wl = inp.wl
    sb = to_np(inp.select_bias) if inp.select_bias is not None else None
    g_logits = to_np(mids["logits"])
    g_ids = to_np(mids["topk_ids"])
    g_w = to_np(mids["topk_w"])
    # (i) the oracle's top-k on the GPU's logits (+ the mode-0 offset the kernel adds)
    l_in = g_logits + (to_np(inp.logit_bias)[None] if (inp.logit_bias is not None and wl.mode == 0) else 0)
    ids_i, w_i = oracle_route_from_logits(l_in, wl, sb)
    assert np.array_equal(g_ids, ids_i), "topk_ids differ from the oracle's top-k of the GPU logits"
    assert np.abs(g_w - w_i).max() <= TOPK_W_RTOL * max(1.0, np.abs(w_i).max())
    # (ii) the oracle's own float64 routing
    l_ref = oracle_logits(inp)
    assert np.abs(l_in - l_ref).max() <= 1e-4 * max(1.0, np.abs(l_ref).max())
    ids_o, w_o = oracle_route_from_logits(l_ref, wl, sb)
    assert np.array_equal(g_ids, ids_o), "topk_ids differ from the oracle's float64 routing"
    # align
    B, mp = mids["block_m"], mids["max_padded"]
    sid, eid, total, counts = O.moe_align(ids_o, B, wl.E, max_padded=mp)
    assert int(mids["num_post_padded"].item()) == total
    assert np.array_equal(to_np(mids["counts"]), counts)
    assert np.array_equal(to_np(mids["sorted_ids"]), sid)
    assert np.array_equal(to_np(mids["expert_ids"]), eid)
    return ids_o, w_o


def _oracle_out(inp, ids, w, tokens=None):
    return O.moe_loop(to_np(inp.x), ids, w, weights_for_oracle(inp.W13),
                      weights_for_oracle(inp.W2), tokens=tokens)


# --------------------------------------------------------------------- page examples (fp32)

def test_page_tiny_layer_f32(L):
    x, wg, w1, w3, w2 = mi.page_tiny_layer()
    inp = _to_dev(mi.LayerInputs(mi.TINY_F32, x, wg, torch.cat([w1, w3], 1), w2))
    layer = _layer(L, inp)
    out = layer(inp.x)
    torch.cuda.synchronize()
    mids = layer.intermediates(64)
    assert to_np(mids["counts"]).tolist() == [19, 11, 15, 15, 21, 15, 18, 14]
    ids, w = _check_routing_and_align(inp, mids)
    assert_close(to_np(out), _oracle_out(inp, ids, w), "f32")


@pytest.mark.parametrize("case", mi.PAGE_FUSED_CASES, ids=[c[0] for c in mi.PAGE_FUSED_CASES])
def test_page_fused_cases_f32(L, golden_dir, case):
    import json, os
    g = {c["name"]: c for c in json.load(open(os.path.join(golden_dir, "fused_cases.json")))["cases"]}
    name, T, E, k, bias = case
    x, wg, w1, w3, w2 = mi.page_fused_case(T, E, bias)
    wl = mi.Workload(name, T=T, H=64, I=96, E=E, k=k, dtype="f32")
    inp = _to_dev(mi.LayerInputs(wl, x, wg, torch.cat([w1, w3], 1), w2))
    layer = _layer(L, inp)
    out = layer(inp.x)
    torch.cuda.synchronize()
    mids = layer.intermediates(T)
    assert to_np(mids["counts"]).tolist() == g[name]["loads"]
    assert int(mids["num_post_padded"].item()) == g[name]["padded"]
    ids, w = _check_routing_and_align(inp, mids)
    assert_close(to_np(out), _oracle_out(inp, ids, w), "f32")


def test_page_deepseek_router(L, golden_dir):
    """The §4 toy router through the GPU top-k: x = logits, Wg = identity (fp32, exact)."""
    import json, os
    g = json.load(open(os.path.join(golden_dir, "deepseek_toy_router.json")))
    logits, bias = mi.page_deepseek_toy()
    x = logits.to(DEV).contiguous()
    Wg = torch.eye(16, device=DEV)
    for b, key in ((torch.zeros(16), "ids_no_bias"), (bias, "ids_with_bias")):
        bd = b.to(DEV)
        cfg = L.make_config(4, 16, 8, 16, 4, L.MOE_F32, L.MOE_ROUTE_SIGMOID_GROUPED, True, 2.5,
                            4, 2, None, bd)
        lg = torch.empty(4, 16, device=DEV)
        ids = torch.empty(4, 4, dtype=torch.int32, device=DEV)
        w = torch.empty(4, 4, device=DEV)
        L.moe_route(cfg, x, Wg, lg, ids, w)
        torch.cuda.synchronize()
        assert torch.equal(lg, x)
        assert ids.cpu().tolist() == g[key]
        if key == "ids_with_bias":
            assert np.abs(to_np(w) - np.array(g["weights_right_3dp"])).max() <= 5e-4 + 1e-6
            _, w_ref = O.route_sigmoid_grouped(to_np(logits), 4, 4, 2, to_np(bias), 2.5)
            assert np.abs(to_np(w) - w_ref).max() <= 1e-6


# --------------------------------------------------------------------- align

ALIGN_CASES = [
    # T, k, E, B, skew  (T*k <= 4096: one-CTA kernel; larger: three-kernel path)
    (4, 3, 5, 4, 0.0), (64, 2, 8, 16, 0.0), (1, 4, 128, 128, 0.0), (37, 1, 8, 16, 0.0),
    (512, 8, 128, 128, 1.2), (4096, 1, 512, 64, 0.5), (8192, 8, 128, 128, 0.0),
    (4096, 8, 256, 128, 1.0), (3000, 7, 300, 1, 0.7), (20000, 2, 8, 128, 2.0),
    (2048, 8, 64, 16, 3.0), (100000, 1, 3, 128, 0.0),
]


@pytest.mark.parametrize("T,k,E,B,skew", ALIGN_CASES)
def test_align_bit_exact(L, T, k, E, B, skew):
    ids = mi.random_topk_ids(T, k, E, seed=T * 31 + E, skew=skew)
    mp = L.moe_max_padded_rows(T, k, E, B)
    sid = torch.full((mp,), -7, dtype=torch.int32, device=DEV)
    eid = torch.full((mp // B,), -7, dtype=torch.int32, device=DEV)
    npp = torch.zeros(1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(E, dtype=torch.int32, device=DEV)
    wsb = L.moe_align_workspace_size(T, k, E, B)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=DEV)
    L.moe_align(ids.to(DEV), T, k, E, B, sid, eid, npp, cnt, ws, wsb)
    torch.cuda.synchronize()
    r_sid, r_eid, r_total, r_cnt = O.moe_align(ids.numpy(), B, E, max_padded=mp)
    assert int(npp.item()) == r_total
    assert np.array_equal(cnt.cpu().numpy(), r_cnt)
    assert np.array_equal(sid.cpu().numpy(), r_sid)
    assert np.array_equal(eid.cpu().numpy(), r_eid)


def test_align_page_example(L, golden_dir):
    import json, os
    g = json.load(open(os.path.join(golden_dir, "align_example.json")))
    ids = torch.tensor(g["topk_ids"], dtype=torch.int32, device=DEV)
    sid = torch.empty(16, dtype=torch.int32, device=DEV)
    eid = torch.empty(4, dtype=torch.int32, device=DEV)
    npp = torch.empty(1, dtype=torch.int32, device=DEV)
    mp = L.moe_max_padded_rows(4, 3, 5, 4)
    sid = torch.empty(mp, dtype=torch.int32, device=DEV)
    eid = torch.empty(mp // 4, dtype=torch.int32, device=DEV)
    L.moe_align(ids, 4, 3, 5, 4, sid, eid, npp)
    torch.cuda.synchronize()
    assert int(npp.item()) == g["total"]
    assert sid[:16].cpu().tolist() == g["sorted_ids"]
    assert eid[:4].cpu().tolist() == g["expert_ids"]


def test_align_bad_expert_id_is_skipped_and_flagged(L):
    ids = torch.tensor([[0, 1], [2, 9], [1, 0]], dtype=torch.int32, device=DEV)  # 9 >= E=4
    mp = L.moe_max_padded_rows(3, 2, 4, 4)
    sid = torch.empty(mp, dtype=torch.int32, device=DEV)
    eid = torch.empty(mp // 4, dtype=torch.int32, device=DEV)
    npp = torch.empty(1, dtype=torch.int32, device=DEV)
    L.moe_device_status(True)
    L.moe_align(ids, 3, 2, 4, 4, sid, eid, npp)
    torch.cuda.synchronize()
    assert L.moe_device_status(True) == 1
    s = sid.cpu().numpy()
    assert 3 not in s.tolist()          # the bad row is never scattered
    assert sorted(x for x in s.tolist() if x < 6) == [0, 1, 2, 4, 5]


# --------------------------------------------------------------------- router

ROUTE_CASES = [
    # name, T, H, E, k, dtype, mode, renorm, scale, G, tg, logit_bias_std, select_bias_std
    ("softmax-E8", 300, 256, 8, 2, "bf16", 0, True, 1.0, 1, 1, 0.0, 0.0),
    ("softmax-E128-offset", 500, 512, 128, 8, "bf16", 0, True, 1.0, 1, 1, 1.5, 0.0),
    ("softmax-norenorm", 200, 128, 32, 4, "bf16", 0, False, 1.0, 1, 1, 0.0, 0.0),
    ("grouped-E256", 300, 512, 256, 8, "bf16", 1, True, 2.5, 8, 4, 0.0, 0.05),
    ("grouped-E64-noscale", 129, 256, 64, 6, "bf16", 1, True, 1.0, 8, 3, 0.0, 0.1),
    ("softmax-E512-simt", 77, 128, 512, 4, "bf16", 0, True, 1.0, 1, 1, 0.0, 0.0),
    ("softmax-E40-f32", 90, 64, 40, 3, "f32", 0, True, 1.0, 1, 1, 0.0, 0.0),
    ("softmax-E300-tiles", 200, 128, 300, 4, "bf16", 0, True, 1.0, 1, 1, 0.0, 0.0),
    ("softmax-f32-tiles", 300, 64, 40, 3, "f32", 0, True, 1.0, 1, 1, 0.0, 0.0),
    ("grouped-decode-T3", 3, 256, 256, 8, "bf16", 1, True, 2.5, 8, 4, 0.0, 0.05),
    ("grouped-E16-f32", 60, 64, 16, 4, "f32", 1, True, 2.5, 4, 2, 0.0, 0.5),
]


@pytest.mark.parametrize("case", ROUTE_CASES, ids=[c[0] for c in ROUTE_CASES])
def test_route_parity(L, case):
    name, T, H, E, k, dt, mode, renorm, scale, G, tg, lbs, sbs = case
    wl = mi.Workload(name, T=T, H=H, I=8, E=E, k=k, dtype=dt, mode=mode, renormalize=renorm,
                     scale=scale, n_group=G, topk_group=tg, logit_bias_std=lbs,
                     select_bias_std=sbs, seed=zlib.crc32(name.encode()) % 1000)
    inp = mi.make_layer(wl, "cpu")
    enforce_margins(inp)
    inp = _to_dev(inp)
    cfg = L.make_config(T, H, 8, E, k, L.MOE_BF16 if dt == "bf16" else L.MOE_F32, mode, renorm,
                        scale, G, tg, inp.logit_bias, inp.select_bias)
    lg = torch.empty(T, E, device=DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, device=DEV)
    L.moe_route(cfg, inp.x, inp.Wg, lg, ids, w)
    torch.cuda.synchronize()
    mids = {"logits": lg, "topk_ids": ids, "topk_w": w}
    sb = to_np(inp.select_bias) if inp.select_bias is not None else None
    l_in = to_np(lg) + (to_np(inp.logit_bias)[None] if inp.logit_bias is not None else 0)
    ids_i, w_i = oracle_route_from_logits(l_in, wl, sb)
    assert np.array_equal(to_np(ids), ids_i)
    assert np.abs(to_np(w) - w_i).max() <= TOPK_W_RTOL * max(1.0, np.abs(w_i).max())
    l_ref = oracle_logits(inp)
    assert np.abs(l_in - l_ref).max() <= 1e-4 * max(1.0, np.abs(l_ref).max())
    ids_o, _ = oracle_route_from_logits(l_ref, wl, sb)
    assert np.array_equal(to_np(mids["topk_ids"]), ids_o)


@pytest.mark.parametrize("mode", [0, 1])
def test_route_exact_ties_go_to_lower_ids(L, mode):
    T, H, E, k = 5, 64, 32, 4
    x = torch.zeros(T, H, device=DEV, dtype=torch.bfloat16)
    Wg = torch.randn(E, H, device=DEV).to(torch.bfloat16)
    cfg = L.make_config(T, H, 8, E, k, L.MOE_BF16, mode, True, 1.0, 4 if mode else 1,
                        2 if mode else 1)
    lg = torch.empty(T, E, device=DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, device=DEV)
    L.moe_route(cfg, x, Wg, lg, ids, w)
    torch.cuda.synchronize()
    assert ids.cpu().tolist() == [[0, 1, 2, 3]] * T
    assert torch.allclose(w.cpu(), torch.full((T, k), 0.25))


# --------------------------------------------------------------------- whole layer, bf16

LAYER_CASES = [
    mi.Workload("bf16-basic", T=200, H=256, I=384, E=8, k=2, dtype="bf16", seed=11),
    mi.Workload("bf16-ragged", T=300, H=320, I=320, E=16, k=4, dtype="bf16", seed=12),
    mi.Workload("bf16-decode-T1", T=1, H=2880, I=2880, E=128, k=4, dtype="bf16", seed=13),
    mi.Workload("bf16-grouped", T=256, H=512, I=256, E=64, k=8, dtype="bf16",
                mode=mi.ROUTE_SIGMOID_GROUPED, scale=2.5, n_group=8, topk_group=4,
                select_bias_std=0.05, seed=14),
    mi.Workload("bf16-skewed", T=600, H=256, I=256, E=32, k=4, dtype="bf16",
                logit_bias_std=1.5, seed=15),
    mi.Workload("bf16-top1", T=37, H=128, I=192, E=8, k=1, dtype="bf16", seed=16),
    # decode above the small-batch limit: the decode tensor-core kernel (weights as the
    # 128-row operand) over ragged K and N; then tiles nearly full (three experts, 256 rows),
    # where the MMA's N covers up to 128 tile rows
    mi.Workload("bf16-decode-T9", T=9, H=320, I=448, E=8, k=4, dtype="bf16", seed=18),
    mi.Workload("bf16-decode-full-tiles", T=128, H=256, I=320, E=3, k=2, dtype="bf16", seed=21),
    # small batches (CUDA-core grouped GEMMs): passes of two rows, the second case with K and
    # N off the 256-element step
    mi.Workload("bf16-decode-T2", T=2, H=2880, I=2880, E=32, k=4, dtype="bf16", seed=19),
    mi.Workload("bf16-decode-T2-ragged", T=2, H=1000, I=776, E=4, k=2, dtype="bf16", seed=20),
    # decode batches route through the one-CTA top-k + align kernel at every expert count:
    # 8 experts a lane (grouped sigmoid, E = 256) and 16 (E = 300)
    mi.Workload("bf16-decode-grouped-E256", T=3, H=256, I=256, E=256, k=8, dtype="bf16",
                mode=mi.ROUTE_SIGMOID_GROUPED, scale=2.5, n_group=8, topk_group=4,
                select_bias_std=0.05, seed=24),
    mi.Workload("bf16-decode-E300", T=2, H=128, I=128, E=300, k=4, dtype="bf16", seed=25),
    mi.Workload("f32-ragged", T=100, H=72, I=88, E=6, k=3, dtype="f32", seed=17),
]


@pytest.mark.parametrize("wl", LAYER_CASES, ids=[w.name for w in LAYER_CASES])
def test_layer_parity(L, wl):
    inp = mi.make_layer(wl, "cpu")
    enforce_margins(inp)
    inp = _to_dev(inp)
    layer = _layer(L, inp)
    out = layer(inp.x)
    torch.cuda.synchronize()
    mids = layer.intermediates(wl.T)
    ids, w = _check_routing_and_align(inp, mids)
    ref = _oracle_out(inp, ids, w)
    assert_close(to_np(out), ref, wl.dtype)
    # y rows: y[r] = w[r] * expert(x[r // k])
    y = to_np(mids["y"])
    n = wl.T * wl.k
    yref = np.zeros_like(y)
    W13, W2 = weights_for_oracle(inp.W13), weights_for_oracle(inp.W2)
    xs = to_np(inp.x)
    for e in np.unique(ids):
        rows = np.nonzero(ids.reshape(-1) == e)[0]
        yref[rows] = O.expert_ffn(xs[rows // wl.k], OM._expert(W13, e), OM._expert(W2, e)) * \
            w.reshape(-1)[rows][:, None]
    assert_close(y[:n], yref, wl.dtype, "y")


ENTRY_CASES = [LAYER_CASES[1],
               mi.Workload("bf16-small-entry", T=2, H=320, I=448, E=8, k=2, dtype="bf16", seed=22)]


@pytest.mark.parametrize("wl", ENTRY_CASES, ids=[w.name for w in ENTRY_CASES])
def test_separate_entry_points_match_forward(L, wl):
    inp = _to_dev(mi.make_layer(wl, "cpu"))
    layer = _layer(L, inp)
    out_fwd = layer(inp.x).clone()
    T, k, E, H, I = wl.T, wl.k, wl.E, wl.H, wl.I
    cfg = layer.config(T)
    assert L.moe_small_batch(cfg) == (T <= 2)
    B = L.moe_block_m(cfg)
    mp = L.moe_max_padded_rows(T, k, E, B)
    lg = torch.empty(T, E, device=DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, device=DEV)
    sid = torch.empty(mp, dtype=torch.int32, device=DEV)
    eid = torch.empty(mp // B, dtype=torch.int32, device=DEV)
    npp = torch.empty(1, dtype=torch.int32, device=DEV)
    act = torch.empty(mp, I, dtype=torch.bfloat16, device=DEV)
    y = torch.empty(T * k, H, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    L.moe_route(cfg, inp.x, inp.Wg, lg, ids, w)
    L.moe_align(ids, T, k, E, B, sid, eid, npp)
    g1b = L.moe_expert_gemm1_workspace_size(cfg, B)
    g1ws = torch.empty(max(g1b, 1), dtype=torch.uint8, device=DEV)
    L.moe_expert_gemm1(cfg, inp.x, inp.W13, sid, eid, npp, B, act, g1ws, g1b)
    g2b = L.moe_expert_gemm2_workspace_size(cfg, B)
    g2ws = torch.empty(max(g2b, 1), dtype=torch.uint8, device=DEV)
    L.moe_expert_gemm2(cfg, act, inp.W2, sid, eid, npp, B, w, y, g2ws, g2b)
    L.moe_combine(y, T, k, H, L.MOE_BF16, out)
    torch.cuda.synchronize()
    assert torch.equal(out, out_fwd)
    # the bf16 GEMM1 split in its two public halves gives the same act
    xs = torch.empty(mp, H, dtype=torch.bfloat16, device=DEV)
    act2 = torch.empty_like(act)
    L.moe_gather_rows(inp.x, sid, npp, T, k, H, L.MOE_BF16, xs)
    gb = L.moe_expert_gemm1_gathered_workspace_size(cfg, B)
    gws = torch.empty(max(gb, 1), dtype=torch.uint8, device=DEV)
    L.moe_expert_gemm1_gathered(cfg, xs, inp.W13, sid, eid, npp, B, act2, gws, gb)
    torch.cuda.synchronize()
    real = (sid < T * k).nonzero().flatten()
    assert torch.equal(act2[real], act[real])
    assert torch.equal(xs[real], inp.x[(sid[real] // k).long()])
    wsb = L.moe_grouped_swiglu_workspace_size(cfg, B)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    y2 = torch.empty_like(y)
    L.moe_grouped_swiglu(cfg, inp.x, inp.W13, inp.W2, sid, eid, npp, B, w, y2, ws, ws.numel())
    torch.cuda.synchronize()
    assert torch.equal(y2, y)


@pytest.mark.parametrize("dtype", ["bf16", "f32", "fp8", "bf16-small", "fp8-small"])
def test_tile_boundaries_and_sentinels(L, dtype):
    """Experts with 0, 1, B-1, B, B+1, 2B-1, 2B, 2B+1 rows; padding rows of act are never
    written (canary survives); every row of y is written (canary gone). "fp8": bf16
    activations with FP8 E4M3 expert weights. "-small": a few rows, which the small-batch
    kernels take (bf16: experts with 0 and 2 rows; FP8: 0, 1, 2 and 5, the last in two
    passes)."""
    small = dtype.endswith("-small")
    dtype = dtype.replace("-small", "")
    fp8 = dtype == "fp8"
    dtype = "bf16" if fp8 else dtype
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    B = 128 if dtype == "bf16" else 16
    if small:
        loads = [0, 1, 2, 5] if fp8 else [0, 2]
    else:
        loads = [0, 1, B - 1, B, B + 1, 2 * B - 1, 2 * B, 2 * B + 1]
    E, k = len(loads), 1
    T = sum(loads)
    H, I = 256, 192
    g = torch.Generator().manual_seed(5)
    ids = torch.tensor([e for e, c in enumerate(loads) for _ in range(c)], dtype=torch.int32)
    ids = ids[torch.randperm(T, generator=g)].view(T, 1)
    w = torch.rand(T, 1, generator=g) + 0.5
    x = torch.randn(T, H, generator=g).to(tdt)
    W13 = (torch.randn(E, 2 * I, H, generator=g) / H ** 0.5).to(tdt)
    W2 = (torch.randn(E, H, I, generator=g) / I ** 0.5).to(tdt)
    sc = {}
    if fp8:
        (W13, s13), (W2, s2) = mi.quantize_fp8_w13(W13), mi.quantize_fp8_blocks(W2)
        sc = dict(w13_scale=s13.to(DEV), w2_scale=s2.to(DEV))
    xd, W13d, W2d, idsd, wd = (t.to(DEV) for t in (x, W13, W2, ids, w))
    cfg = L.make_config(T, H, I, E, k, L.MOE_BF16 if dtype == "bf16" else L.MOE_F32, **sc)
    assert L.moe_small_batch(cfg) == small
    mp = L.moe_max_padded_rows(T, k, E, B)
    sid = torch.empty(mp, dtype=torch.int32, device=DEV)
    eid = torch.empty(mp // B, dtype=torch.int32, device=DEV)
    npp = torch.empty(1, dtype=torch.int32, device=DEV)
    act = torch.full((mp, I), float("nan"), dtype=tdt, device=DEV)
    y = torch.full((T * k, H), float("nan"), dtype=tdt, device=DEV)
    out = torch.empty(T, H, dtype=tdt, device=DEV)
    L.moe_align(idsd, T, k, E, B, sid, eid, npp)
    g1b = L.moe_expert_gemm1_workspace_size(cfg, B)
    g1ws = torch.empty(max(g1b, 1), dtype=torch.uint8, device=DEV)
    L.moe_expert_gemm1(cfg, xd, W13d, sid, eid, npp, B, act, g1ws, g1b)
    g2b = L.moe_expert_gemm2_workspace_size(cfg, B)
    g2ws = torch.empty(max(g2b, 1), dtype=torch.uint8, device=DEV)
    L.moe_expert_gemm2(cfg, act, W2d, sid, eid, npp, B, wd, y, g2ws, g2b)
    L.moe_combine(y, T, k, H, cfg.dtype, out)
    torch.cuda.synchronize()
    s = sid.cpu().numpy()
    total = int(npp.item())
    valid = s < T * k
    a = act.float().cpu().numpy()
    assert np.all(np.isfinite(a[valid])), "a real row of act was not written"
    assert np.all(np.isnan(a[~valid])), "a padding row of act was written"
    assert np.all(np.isfinite(y.float().cpu().numpy())), "a row of y was not written"
    assert total == sum((c + B - 1) // B * B for c in loads)
    if fp8:
        w13o = O.dequant_w13(W13.numpy(), s13.double().numpy())
        w2o = O.dequant_blockwise(W2.numpy(), s2.double().numpy())
    else:
        w13o, w2o = weights_for_oracle(W13), weights_for_oracle(W2)
    ref = O.moe_loop(to_np(x), ids.numpy(), to_np(w), w13o, w2o)
    assert_close(to_np(out), ref, dtype)


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
def test_small_batch_repeated_expert(L, fp8):
    """One token that lists an expert twice (valid input for the align and grouped GEMM entry
    points): that expert's tile holds more real rows than there are tokens, so the
    small-batch kernels (one row a pass at T = 1) stream its weights in two passes; y and the
    combined output equal the oracle's."""
    T, k, E, H, I = 1, 3, 4, 320, 448
    g = torch.Generator().manual_seed(23)
    ids = torch.tensor([[2, 2, 0]], dtype=torch.int32)
    w = torch.rand(T, k, generator=g) + 0.5
    x = torch.randn(T, H, generator=g).bfloat16()
    W13 = (torch.randn(E, 2 * I, H, generator=g) / H ** 0.5).bfloat16()
    W2 = (torch.randn(E, H, I, generator=g) / I ** 0.5).bfloat16()
    sc = {}
    if fp8:
        (W13, s13), (W2, s2) = mi.quantize_fp8_w13(W13), mi.quantize_fp8_blocks(W2)
        sc = dict(w13_scale=s13.to(DEV), w2_scale=s2.to(DEV))
        w13o = O.dequant_w13(W13.numpy(), s13.double().numpy())
        w2o = O.dequant_blockwise(W2.numpy(), s2.double().numpy())
    else:
        w13o, w2o = weights_for_oracle(W13), weights_for_oracle(W2)
    cfg = L.make_config(T, H, I, E, k, L.MOE_BF16, **sc)
    assert L.moe_small_batch(cfg)
    B = 128
    mp = L.moe_max_padded_rows(T, k, E, B)
    sid = torch.empty(mp, dtype=torch.int32, device=DEV)
    eid = torch.empty(mp // B, dtype=torch.int32, device=DEV)
    npp = torch.empty(1, dtype=torch.int32, device=DEV)
    y = torch.full((T * k, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(L.moe_grouped_swiglu_workspace_size(cfg, B), dtype=torch.uint8, device=DEV)
    L.moe_align(ids.to(DEV), T, k, E, B, sid, eid, npp)
    L.moe_grouped_swiglu(cfg, x.to(DEV), W13.to(DEV), W2.to(DEV), sid, eid, npp, B, w.to(DEV), y,
                         ws, ws.numel())
    L.moe_combine(y, T, k, H, L.MOE_BF16, out)
    torch.cuda.synchronize()
    xs = to_np(x)
    yref = np.stack([O.expert_ffn(xs, OM._expert(w13o, e), OM._expert(w2o, e))[0] * w[0, j].item()
                     for j, e in enumerate(ids[0].tolist())])
    assert_close(to_np(y), yref, "bf16", "y")
    ref = O.moe_loop(xs, ids.numpy(), to_np(w), w13o, w2o)
    assert_close(to_np(out), ref, "bf16")


def test_stalled_pipeline_times_out_with_a_status(L):
    """A pipeline wait that nothing satisfies gives up after its limit (about 2 s): the kernel
    returns, the status word reads 2, and the context still runs a layer correctly."""
    import time
    L.moe_device_status(True)
    t0 = time.time()
    L.moe_selftest_wait_timeout()
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert L.moe_device_status(True) == 2
    assert 1.5 < dt < 30
    wl = mi.Workload("after-timeout", T=64, H=128, I=128, E=8, k=2, dtype="bf16", seed=71)
    inp = mi.make_layer(wl, "cpu")
    enforce_margins(inp)
    inp = _to_dev(inp)
    out = _layer(L, inp)(inp.x)
    torch.cuda.synchronize()
    ids, w = oracle_route_from_logits(oracle_logits(inp), wl)
    assert_close(to_np(out), _oracle_out(inp, ids, w), "bf16")
    assert L.moe_device_status(True) == 0


def test_all_tokens_to_one_expert(L):
    T, H, I, E, k = 700, 256, 256, 16, 2
    g = torch.Generator().manual_seed(9)
    ids = torch.stack([torch.full((T,), 3), torch.randint(4, E, (T,), generator=g)], 1).int()
    w = torch.rand(T, k, generator=g)
    x = torch.randn(T, H, generator=g).bfloat16()
    W13 = (torch.randn(E, 2 * I, H, generator=g) / H ** 0.5).bfloat16()
    W2 = (torch.randn(E, H, I, generator=g) / I ** 0.5).bfloat16()
    cfg = L.make_config(T, H, I, E, k, L.MOE_BF16)
    B = 128
    mp = L.moe_max_padded_rows(T, k, E, B)
    sid = torch.empty(mp, dtype=torch.int32, device=DEV)
    eid = torch.empty(mp // B, dtype=torch.int32, device=DEV)
    npp = torch.empty(1, dtype=torch.int32, device=DEV)
    y = torch.empty(T * k, H, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(L.moe_grouped_swiglu_workspace_size(cfg, B), dtype=torch.uint8, device=DEV)
    xd, W13d, W2d = x.to(DEV), W13.to(DEV), W2.to(DEV)
    L.moe_align(ids.to(DEV), T, k, E, B, sid, eid, npp)
    L.moe_grouped_swiglu(cfg, xd, W13d, W2d, sid, eid, npp, B, w.to(DEV), y, ws, ws.numel())
    L.moe_combine(y, T, k, H, L.MOE_BF16, out)
    torch.cuda.synchronize()
    ref = O.moe_loop(to_np(x), ids.numpy(), to_np(w), weights_for_oracle(W13), weights_for_oracle(W2))
    assert_close(to_np(out), ref, "bf16")


@pytest.mark.parametrize("T", [256, 48])  # the CTA-pair GEMMs; the decode tensor-core GEMMs
def test_cuda_graph_capture_and_replay(L, T):
    wl = mi.Workload("graph", T=T, H=256, I=256, E=16, k=4, dtype="bf16", seed=21)
    inp = _to_dev(mi.make_layer(wl, "cpu"))
    layer = _layer(L, inp)
    x_static = inp.x.clone()
    out_static = torch.empty_like(x_static)
    layer(x_static, out_static)          # first call sets up the workspace / kernels
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            layer(x_static, out_static)
    torch.cuda.current_stream().wait_stream(s)
    for seed in (1, 2):
        xn = torch.randn(wl.T, wl.H, generator=torch.Generator().manual_seed(seed)).bfloat16()
        x_static.copy_(xn.to(DEV))
        graph.replay()
        torch.cuda.synchronize()
        eager = layer(x_static.clone())
        torch.cuda.synchronize()
        assert torch.equal(out_static, eager)


# --------------------------------------------------------------------- expert parallelism

@pytest.mark.parametrize("dtype,variant,T", [("bf16", "half", 300), ("bf16", "perm", 300),
                                             ("f32", "half", 300), ("fp8", "perm", 300),
                                             ("bf16", "half", 2), ("fp8", "perm", 6),
                                             ("bf16", "half", 40), ("fp8", "perm", 40)])
def test_expert_map(L, dtype, variant, T):
    """Odd experts held elsewhere (map -1), or local experts stored in permuted weight slots:
    the layer equals the oracle with the same expert_map; tiles carry the mapped labels.
    "fp8": the permuted slots hold FP8 codes whose block scales are permuted with them."""
    fp8 = dtype == "fp8"
    dtype = "bf16" if fp8 else dtype
    H, I = (256, 256) if dtype == "bf16" else (64, 96)
    wl = mi.Workload("ep", T=T, H=H, I=I, E=16, k=4, dtype=dtype, seed=31)
    inp = mi.make_layer(wl, "cpu")
    enforce_margins(inp)
    E = wl.E
    if variant == "half":
        emap = torch.tensor([e if e % 2 == 0 else -1 for e in range(E)], dtype=torch.int32)
        W13, W2 = inp.W13, inp.W2
    else:
        emap = torch.tensor([(5 * e + 3) % E for e in range(E)], dtype=torch.int32)
        W13, W2 = torch.empty_like(inp.W13), torch.empty_like(inp.W2)
        W13[emap.long()], W2[emap.long()] = inp.W13, inp.W2
    sc = {}
    if fp8:  # quantise the stored (slot-ordered) weights; the oracle takes their exact values
        (W13, s13), (W2, s2) = mi.quantize_fp8_w13(W13), mi.quantize_fp8_blocks(W2)
        sc = dict(w13_scale=s13.to(DEV), w2_scale=s2.to(DEV))
    dev = _to_dev(mi.LayerInputs(wl, inp.x, inp.Wg, W13, W2))
    from routing_grouped_gemm_router_gb300.layer import MoELayer
    layer = MoELayer(dev.Wg, dev.W13, dev.W2, wl.k, expert_map=emap.to(DEV), **sc)
    out = layer(dev.x)
    torch.cuda.synchronize()
    mids = layer.intermediates(wl.T)
    ids, w = O.route_softmax(oracle_logits(inp), wl.k)
    assert np.array_equal(to_np(mids["topk_ids"]), ids)
    B, mp = mids["block_m"], mids["max_padded"]
    _, eid, _, _ = O.moe_align(ids, B, E, max_padded=mp)
    assert np.array_equal(to_np(mids["expert_ids"]), O.apply_expert_map(eid, emap.numpy()))
    if fp8:
        W13o = O.dequant_w13(W13.numpy(), s13.double().numpy())
        W2o = O.dequant_blockwise(W2.numpy(), s2.double().numpy())
    else:
        W13o, W2o = weights_for_oracle(W13), weights_for_oracle(W2)
    ref = O.moe_loop(to_np(inp.x), ids, w, W13o, W2o, expert_map=emap.numpy())
    assert_close(to_np(out), ref, dtype)
    if variant == "perm" and not fp8:  # same layer as without expert parallelism
        plain = O.moe_loop(to_np(inp.x), ids, w, weights_for_oracle(inp.W13),
                           weights_for_oracle(inp.W2))
        assert_close(to_np(out), plain, dtype)


def test_combine_local_skips_and_flags_bad_expert_id(L):
    """A slot whose id lies outside [0, E) is left out of the sum (its y row was never
    computed) and sets device status 1; remote slots (map -1) are left out silently."""
    T, k, E, H = 3, 2, 4, 16
    ids = torch.tensor([[0, 1], [2, 9], [3, -1]], dtype=torch.int32, device=DEV)
    emap = torch.tensor([0, -1, 2, 3], dtype=torch.int32, device=DEV)
    y = (torch.arange(T * k * H, dtype=torch.float32, device=DEV).view(T * k, H) + 1.0)
    out = torch.full((T, H), -7.0, dtype=torch.float32, device=DEV)
    L.moe_device_status(True)
    L.moe_combine_local(y, ids, emap, E, T, k, H, L.MOE_F32, out)
    torch.cuda.synchronize()
    assert L.moe_device_status(True) == 1
    yc = y.cpu()
    ref = torch.stack([yc[0], yc[2], yc[4]])  # slots (0,1), (1,1), (2,1) dropped
    assert torch.equal(out.cpu(), ref)


# --------------------------------------------------------------------- shared experts

@pytest.mark.parametrize("dtype,T", [("bf16", 200), ("f32", 200), ("bf16", 2), ("bf16", 40)])
def test_shared_expert(L, dtype, T):
    """DeepSeek-style layer with one shared expert (weight 1 on every token), grouped
    sigmoid routing with scale 2.5: equals the oracle with the shared slot appended."""
    H, I = (256, 256) if dtype == "bf16" else (64, 96)
    wl = mi.Workload("shared", T=T, H=H, I=I, E=16, k=4, dtype=dtype,
                     mode=mi.ROUTE_SIGMOID_GROUPED, scale=2.5, n_group=4, topk_group=2,
                     select_bias_std=0.05, seed=41)
    inp = mi.make_layer(wl, "cpu")
    enforce_margins(inp)
    g = torch.Generator().manual_seed(42)
    tdt = inp.W13.dtype
    W13 = torch.cat([inp.W13, (torch.randn(1, 2 * I, H, generator=g) / H ** 0.5).to(tdt)])
    W2 = torch.cat([inp.W2, (torch.randn(1, H, I, generator=g) / I ** 0.5).to(tdt)])
    dev = _to_dev(mi.LayerInputs(wl, inp.x, inp.Wg, W13, W2, None, inp.select_bias))
    from routing_grouped_gemm_router_gb300.layer import MoELayer
    layer = MoELayer(dev.Wg, dev.W13, dev.W2, wl.k, wl.mode, True, wl.scale, wl.n_group,
                     wl.topk_group, None, dev.select_bias, n_shared=1)
    out = layer(dev.x)
    torch.cuda.synchronize()
    mids = layer.intermediates(wl.T)
    ids, w = O.route_sigmoid_grouped(oracle_logits(inp), wl.k, wl.n_group, wl.topk_group,
                                     to_np(inp.select_bias), wl.scale)
    ids, w = O.add_shared_experts(ids, w, wl.E, 1)
    assert np.array_equal(to_np(mids["topk_ids"]), ids)
    assert np.all(to_np(mids["topk_w"])[:, -1] == 1.0)
    ref = O.moe_loop(to_np(inp.x), ids, w, weights_for_oracle(W13), weights_for_oracle(W2))
    assert_close(to_np(out), ref, dtype)


# --------------------------------------------------------------------- fixed-capacity layout

@pytest.mark.parametrize("dtype,with_w", [("bf16", True), ("bf16", False), ("f32", True)])
def test_masked_layout(L, dtype, with_w):
    """Tokens bucketed per expert with a fixed capacity: valid rows equal the oracle's
    masked forward; rows past each count are never written (canary survives)."""
    H, I = (256, 384) if dtype == "bf16" else (64, 96)
    B = 128 if dtype == "bf16" else 16
    wl = mi.Workload("masked", T=150, H=H, I=I, E=8, k=2, dtype=dtype, seed=51)
    inp = mi.make_layer(wl, "cpu")
    ids, w = O.route_softmax(oracle_logits(inp), wl.k)
    cap = -(-int(np.bincount(ids.ravel(), minlength=wl.E).max()) // B) * B + B
    xm, wm, counts, _ = O.dispatch_masked(to_np(inp.x), ids, w, wl.E, cap)
    tdt = inp.x.dtype
    xm_d = torch.tensor(xm, dtype=tdt, device=DEV)
    wm_d = torch.tensor(wm, dtype=torch.float32, device=DEV) if with_w else None
    cnt_d = torch.tensor(counts, dtype=torch.int32, device=DEV)
    y = torch.full((wl.E, cap, H), float("nan"), dtype=tdt, device=DEV)
    cfg = L.make_config(1, H, I, wl.E, 1, L.MOE_BF16 if dtype == "bf16" else L.MOE_F32)
    wsb = L.moe_masked_workspace_size(cfg, cap)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    W13, W2 = inp.W13.to(DEV), inp.W2.to(DEV)
    for rep in range(2):
        L.moe_masked_forward(cfg, xm_d, cnt_d, cap, wm_d, W13, W2, y, ws, wsb)
    torch.cuda.synchronize()
    ref = O.masked_forward(to_np(xm_d), counts, weights_for_oracle(inp.W13),
                           weights_for_oracle(inp.W2), wm if with_w else None)
    got = to_np(y)
    valid = ~np.isnan(ref[:, :, 0])
    assert np.array_equal(valid, np.arange(cap)[None, :] < counts[:, None])
    assert np.all(np.isnan(got[~valid])), "a row past an expert's count was written"
    assert_close(got[valid], ref[valid], dtype)
    # the table alone: identity on valid rows, tiles past a count labelled -1
    n = wl.E * cap
    sid = torch.empty(n, dtype=torch.int32, device=DEV)
    eid = torch.empty(n // B, dtype=torch.int32, device=DEV)
    npp = torch.empty(1, dtype=torch.int32, device=DEV)
    L.moe_masked_table(cnt_d, wl.E, cap, B, sid, eid, npp)
    torch.cuda.synchronize()
    p = np.arange(n)
    exp_sid = np.where((p % cap) < counts[p // cap], p, n)
    t = np.arange(n // B)
    exp_eid = np.where(((t * B) % cap) < counts[(t * B) // cap], (t * B) // cap, -1)
    assert np.array_equal(sid.cpu().numpy(), exp_sid) and int(npp.item()) == n
    assert np.array_equal(eid.cpu().numpy(), exp_eid)


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
def test_masked_layout_capacity_128(L, fp8):
    """Capacity 128 (one tile per expert, the decode case) takes the decode tensor-core
    kernels: empty experts, experts of 1-9 rows and one full tile (128 rows) all match the
    oracle's masked forward, and rows past each count are never written."""
    H, I, E, B = 320, 272, 12, 128
    wl = mi.Workload("masked-128", T=1, H=H, I=I, E=E, k=1, dtype="bf16", seed=53)
    inp = mi.make_layer(wl, "cpu")
    counts = np.array([0, 1, 3, 9, 0, 2, 128, 5, 1, 0, 7, 4], dtype=np.int32)
    g = torch.Generator().manual_seed(54)
    xm = torch.randn(E, B, H, generator=g).bfloat16()
    wm = (torch.rand(E, B, generator=g) + 0.5).numpy()
    W13, W2, sc = inp.W13, inp.W2, {}
    if fp8:
        (W13, s13), (W2, s2) = mi.quantize_fp8_w13(W13), mi.quantize_fp8_blocks(W2)
        sc = dict(w13_scale=s13.to(DEV), w2_scale=s2.to(DEV))
        W13o = O.dequant_w13(W13.numpy(), s13.double().numpy())
        W2o = O.dequant_blockwise(W2.numpy(), s2.double().numpy())
    else:
        W13o, W2o = weights_for_oracle(W13), weights_for_oracle(W2)
    cfg = L.make_config(1, H, I, E, 1, L.MOE_BF16, **sc)
    y = torch.full((E, B, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    wsb = L.moe_masked_workspace_size(cfg, B)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    L.moe_masked_forward(cfg, xm.to(DEV), torch.tensor(counts, device=DEV), B,
                         torch.tensor(wm, device=DEV), W13.to(DEV), W2.to(DEV), y, ws, wsb)
    torch.cuda.synchronize()
    assert L.moe_device_status(True) == 0
    ref = O.masked_forward(to_np(xm), counts, W13o, W2o, wm)
    got = to_np(y)
    valid = np.arange(B)[None, :] < counts[:, None]
    assert np.all(np.isnan(got[~valid])), "a row past an expert's count was written"
    assert_close(got[valid], ref[valid], "bf16")


# --------------------------------------------------------------------- FP8 expert weights

FP8_CASES = [
    # ragged: H = 2.5 scale blocks, I = 2 panels + 16 rows, GEMM2 K = 4.25 k-blocks
    (mi.Workload("fp8-ragged", T=300, H=320, I=272, E=8, k=2, dtype="bf16", seed=61), 0, False),
    # grouped sigmoid router, scale 2.5, one shared expert
    (mi.Workload("fp8-grouped-shared", T=256, H=512, I=384, E=32, k=8, dtype="bf16",
                 mode=mi.ROUTE_SIGMOID_GROUPED, scale=2.5, n_group=8, topk_group=4,
                 select_bias_std=0.05, seed=62), 1, False),
    # scales that are not powers of two: the kernel rounds code * scale to bf16 once
    (mi.Workload("fp8-any-scale", T=200, H=256, I=256, E=16, k=4, dtype="bf16", seed=63), 0, True),
    # decode (small-batch kernels): one token; six tokens on four experts (rows of an expert
    # in two passes) with K off the 512-code step and any scales; three tokens + a shared one;
    # 24 tokens on eight experts (tiles of 2-10 rows: passes of four rows and shorter ones)
    (mi.Workload("fp8-decode", T=1, H=512, I=512, E=64, k=4, dtype="bf16", seed=64), 0, False),
    (mi.Workload("fp8-decode-ragged", T=6, H=1040, I=784, E=4, k=2, dtype="bf16", seed=66), 0,
     True),
    (mi.Workload("fp8-decode-shared", T=3, H=2880, I=1024, E=16, k=4, dtype="bf16", seed=67), 1,
     False),
    (mi.Workload("fp8-decode-T24", T=24, H=320, I=272, E=8, k=2, dtype="bf16", seed=71), 0, True),
    # decode tensor-core kernel (25 to 128 tokens): ragged K and N with any scales; 64 tokens
    # plus a shared expert (a 64-row tile); tiles nearly full (one tile-row slot in GEMM1)
    (mi.Workload("fp8-dec-ragged", T=28, H=320, I=272, E=8, k=2, dtype="bf16", seed=68), 0, True),
    (mi.Workload("fp8-dec-shared", T=64, H=512, I=384, E=32, k=4, dtype="bf16", seed=69), 1,
     False),
    (mi.Workload("fp8-dec-full-tiles", T=128, H=256, I=256, E=3, k=2, dtype="bf16", seed=70), 0,
     False),
]


def _fp8_weights(inp, n_shared, any_scale, seed):
    g = torch.Generator().manual_seed(seed)
    H, I = inp.wl.H, inp.wl.I
    W13, W2 = inp.W13, inp.W2
    if n_shared:
        W13 = torch.cat([W13, (torch.randn(n_shared, 2 * I, H, generator=g) / H ** 0.5).bfloat16()])
        W2 = torch.cat([W2, (torch.randn(n_shared, H, I, generator=g) / I ** 0.5).bfloat16()])
    (c13, s13), (c2, s2) = mi.quantize_fp8_w13(W13), mi.quantize_fp8_blocks(W2)
    if any_scale:
        s13 = s13 * (1.0 + torch.rand(s13.shape, generator=g))
        s2 = s2 * (1.0 + torch.rand(s2.shape, generator=g))
    return c13, s13, c2, s2


@pytest.mark.parametrize("wl,n_shared,any_scale", FP8_CASES, ids=[c[0].name for c in FP8_CASES])
def test_fp8_layer_parity(L, wl, n_shared, any_scale):
    """moe_forward with FP8 E4M3 expert weights and 128 x 128 block scales equals the
    float64 oracle run on the dequantised weights (code * scale)."""
    from routing_grouped_gemm_router_gb300.layer import MoELayer
    inp = mi.make_layer(wl, "cpu")
    enforce_margins(inp)
    c13, s13, c2, s2 = _fp8_weights(inp, n_shared, any_scale, wl.seed)
    d = lambda t: None if t is None else t.to(DEV).contiguous()  # noqa: E731
    layer = MoELayer(d(inp.Wg), d(c13), d(c2), wl.k, wl.mode, wl.renormalize, wl.scale,
                     wl.n_group, wl.topk_group, d(inp.logit_bias), d(inp.select_bias),
                     n_shared=n_shared, w13_scale=d(s13), w2_scale=d(s2))
    kind = (L.MOE_GEMM_SMALL_BATCH if wl.name.startswith("fp8-decode") else
            L.MOE_GEMM_DECODE_TC if wl.name.startswith("fp8-dec-") else L.MOE_GEMM_PAIR_TC)
    assert L.moe_gemm_kernel(layer.config(wl.T)) == kind
    out = layer(d(inp.x))
    torch.cuda.synchronize()
    mids = layer.intermediates(wl.T)
    sb = to_np(inp.select_bias) if inp.select_bias is not None else None
    ids, w = oracle_route_from_logits(oracle_logits(inp), wl, sb)
    if n_shared:
        ids, w = O.add_shared_experts(ids, w, wl.E, n_shared)
    assert np.array_equal(to_np(mids["topk_ids"]), ids)
    w13o = O.dequant_w13(c13.numpy(), s13.double().numpy())
    w2o = O.dequant_blockwise(c2.numpy(), s2.double().numpy())
    ref = O.moe_loop(to_np(inp.x), ids, w, w13o, w2o)
    assert_close(to_np(out), ref, "bf16")
    if not any_scale:
        # power-of-two scales: the dequantised weights are exact in bf16, so the result is
        # the bf16 layer's on those weights: bit for bit on the tensor cores (codes scaled
        # before the products); the small-batch kernels scale 16-code partial sums instead,
        # which agrees to within rounding
        layer_bf = MoELayer(d(inp.Wg), d(torch.tensor(w13o).bfloat16()),
                            d(torch.tensor(w2o).bfloat16()), wl.k, wl.mode, wl.renormalize,
                            wl.scale, wl.n_group, wl.topk_group, d(inp.logit_bias),
                            d(inp.select_bias), n_shared=n_shared)
        out_bf = layer_bf(d(inp.x))
        torch.cuda.synchronize()
        if L.moe_small_batch(layer.config(wl.T)):
            assert_close(to_np(out), to_np(out_bf).astype(np.float64), "bf16")
        else:
            assert torch.equal(out_bf, out)


def test_fp8_masked_layout(L):
    """The fixed-capacity layout with FP8 weights: valid rows equal the oracle's masked
    forward on the dequantised weights; rows past each count are never written."""
    H, I, E, B = 256, 384, 8, 128
    wl = mi.Workload("fp8-masked", T=150, H=H, I=I, E=E, k=2, dtype="bf16", seed=65)
    inp = mi.make_layer(wl, "cpu")
    ids, w = O.route_softmax(oracle_logits(inp), wl.k)
    cap = -(-int(np.bincount(ids.ravel(), minlength=E).max()) // B) * B + B
    xm, wm, counts, _ = O.dispatch_masked(to_np(inp.x), ids, w, E, cap)
    c13, s13, c2, s2 = _fp8_weights(inp, 0, False, 65)
    s13d, s2d = s13.to(DEV), s2.to(DEV)   # the config points at these: keep them alive
    cfg = L.make_config(1, H, I, E, 1, L.MOE_BF16, w13_scale=s13d, w2_scale=s2d)
    xm_d = torch.tensor(xm, dtype=torch.bfloat16, device=DEV)
    y = torch.full((E, cap, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    wsb = L.moe_masked_workspace_size(cfg, cap)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    L.moe_masked_forward(cfg, xm_d, torch.tensor(counts, dtype=torch.int32, device=DEV), cap,
                         torch.tensor(wm, dtype=torch.float32, device=DEV), c13.to(DEV),
                         c2.to(DEV), y, ws, wsb)
    torch.cuda.synchronize()
    ref = O.masked_forward(to_np(xm_d), counts, O.dequant_w13(c13.numpy(), s13.double().numpy()),
                           O.dequant_blockwise(c2.numpy(), s2.double().numpy()), wm)
    got = to_np(y)
    valid = ~np.isnan(ref[:, :, 0])
    assert np.all(np.isnan(got[~valid])), "a row past an expert's count was written"
    assert_close(got[valid], ref[valid], "bf16")


@pytest.mark.parametrize("any_scale", [False, True], ids=["pow2-scales", "any-scales"])
def test_dequant_fp8_weights(L, any_scale):
    """moe_dequant_fp8_weights: every weight of W13 and W2 is code * block scale as bf16 —
    equal to the oracle's float64 dequantisation for power-of-two scales (the products are
    exact), within one bf16 rounding of it otherwise; experts whose count is 0 are not
    written."""
    wl = mi.Workload("dq", T=64, H=384, I=272, E=4, k=2, dtype="bf16", seed=81)
    inp = mi.make_layer(wl, "cpu")
    c13, s13, c2, s2 = _fp8_weights(inp, 1, any_scale, wl.seed)
    E, H, I = wl.E + 1, wl.H, wl.I
    s13d, s2d = s13.to(DEV), s2.to(DEV)  # the config holds their addresses
    cfg = L.make_config(wl.T, H, I, wl.E, wl.k, L.MOE_BF16, n_shared=1, w13_scale=s13d,
                        w2_scale=s2d)
    counts = torch.tensor([3, 0, 5, 1, 2], dtype=torch.int32, device=DEV)
    for matrix, codes, ref in ((1, c13, O.dequant_w13(c13.numpy(), s13.double().numpy())),
                               (2, c2, O.dequant_blockwise(c2.numpy(), s2.double().numpy()))):
        out = torch.full(tuple(codes.shape), float("nan"), dtype=torch.bfloat16, device=DEV)
        L.moe_dequant_fp8_weights(cfg, matrix, codes.to(DEV), None, out)
        got = to_np(out)
        if any_scale:
            assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref))
        else:
            assert np.array_equal(got, ref)
        skip = torch.full_like(out, float("nan"))
        L.moe_dequant_fp8_weights(cfg, matrix, codes.to(DEV), counts, skip)
        torch.cuda.synchronize()
        live = (counts > 0).cpu()
        assert torch.equal(skip[live.to(DEV)], out[live.to(DEV)])
        assert torch.isnan(skip[~live.to(DEV)].float()).all()
