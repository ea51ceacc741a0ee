"""Parity at the full workload sizes, in the launch configuration the benchmark times.

Each layer is drawn on the GPU (seeded), routed, aligned and run through moe_forward.
Routing and the indirection table are checked bit-exactly for every token; the layer
output is checked on a sample of tokens (tokens of the hottest and of the least-loaded
non-empty expert among them), and the grouped GEMMs' output y on the first and last routed
row of every active expert, each recomputed by the float64 oracle.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle as O
from _helpers import (LazyExperts, LazyExpertsF64, LazyFp8Experts, assert_close, enforce_margins, oracle_logits,
                      oracle_route_from_logits, sample_tokens, to_np)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
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
    assert _lib.moe_device_status(True) == 0


CASES = [(mi.MIXTRAL, 48), (mi.QWEN3, 48), (mi.DSV3, 16)] + \
        [(mi.GPTOSS.with_T(T), T) for T in mi.GPTOSS_T]


@pytest.mark.parametrize("wl,n_sample", CASES, ids=[c[0].name for c in CASES])
def test_full_size_parity(L, wl, n_sample):
    from routing_grouped_gemm_router_gb300.layer import MoELayer
    inp = mi.make_layer(wl, DEV)
    redraws = enforce_margins(inp)
    layer = MoELayer(inp.Wg, inp.W13, inp.W2, wl.k, wl.mode, wl.renormalize, wl.scale,
                     wl.n_group, wl.topk_group, inp.logit_bias, inp.select_bias)
    out = layer(inp.x)
    torch.cuda.synchronize()
    mids = layer.intermediates(wl.T)

    # routing: all tokens, both readings
    sb = to_np(inp.select_bias) if inp.select_bias is not None else None
    g_logits = to_np(mids["logits"])
    l_in = g_logits + (to_np(inp.logit_bias)[None] if inp.logit_bias is not None else 0)
    g_ids = to_np(mids["topk_ids"])
    ids_i, w_i = oracle_route_from_logits(l_in, wl, sb)
    assert np.array_equal(g_ids, ids_i)
    assert np.abs(to_np(mids["topk_w"]) - w_i).max() <= 2e-5 * max(1.0, np.abs(w_i).max())
    l_ref = oracle_logits(inp)
    ids_o, w_o = oracle_route_from_logits(l_ref, wl, sb)
    assert np.array_equal(g_ids, ids_o), f"routing differs ({redraws} margin redraws)"

    # align: bit-exact
    B, mp = mids["block_m"], mids["max_padded"]
    sid, eid, total, counts = O.moe_align(ids_o, B, wl.E, max_padded=mp)
    assert int(mids["num_post_padded"].item()) == total
    assert np.array_equal(to_np(mids["counts"]), counts)
    assert np.array_equal(to_np(mids["sorted_ids"]), sid)
    assert np.array_equal(to_np(mids["expert_ids"]), eid)
    if wl.name.startswith("qwen3"):
        assert (counts == 0).any(), "the skewed workload should leave some experts empty"

    # output: sampled tokens against the float64 oracle
    toks = sample_tokens(ids_o, n_sample, seed=wl.seed)
    ref = O.moe_loop(to_np(inp.x[torch.as_tensor(toks, device=DEV)]),
                     ids_o[toks], w_o[toks], LazyExperts(inp.W13), LazyExperts(inp.W2))
    got = to_np(out[torch.as_tensor(toks, device=DEV)])
    assert_close(got, ref, wl.dtype)
    assert torch.isfinite(out.float()).all()

    # y: for every active expert its first and last routed rows (its first and last m-tile),
    # each a full row of H outputs against the oracle's single-slot layer (w_r times the
    # expert's FFN of the token), so an error confined to one weight panel of any expert,
    # in either grouped GEMM, shows
    k = wl.k
    flat = ids_o.ravel()
    rows = []
    for e in np.unique(flat):
        r_e = np.nonzero(flat == e)[0]
        rows += sorted({int(r_e[0]), int(r_e[-1])})
    rows = np.array(rows)
    t_sel = rows // k
    y_ref = O.moe_loop(to_np(inp.x[torch.as_tensor(t_sel, device=DEV)]), flat[rows][:, None],
                       w_o.ravel()[rows][:, None], LazyExperts(inp.W13), LazyExperts(inp.W2))
    y_got = to_np(mids["y"][torch.as_tensor(rows, device=DEV)])
    assert_close(y_got, y_ref, wl.dtype)


FP8_CASES = [(mi.DSV3, 16), (mi.GPTOSS.with_T(1), 1), (mi.GPTOSS.with_T(16), 16),
             (mi.GPTOSS.with_T(128), 32)]


@pytest.mark.parametrize("wl,n_sample", FP8_CASES, ids=[c[0].name + "-fp8" for c in FP8_CASES])
def test_full_size_fp8_parity(L, wl, n_sample):
    """Full-size layers with FP8 E4M3 expert weights (128 x 128 block scales, drawn by
    quantising the seeded bf16 weights): routing bit-exact, sampled tokens against the
    oracle on the dequantised weights."""
    from routing_grouped_gemm_router_gb300.layer import MoELayer
    inp = mi.make_layer(wl, DEV)
    enforce_margins(inp)
    c13, s13 = mi.quantize_fp8_w13(inp.W13)
    c2, s2 = mi.quantize_fp8_blocks(inp.W2)
    inp.W13 = inp.W2 = None
    torch.cuda.empty_cache()
    layer = MoELayer(inp.Wg, c13, c2, wl.k, wl.mode, wl.renormalize, wl.scale, wl.n_group,
                     wl.topk_group, inp.logit_bias, inp.select_bias, w13_scale=s13, w2_scale=s2)
    out = layer(inp.x)
    torch.cuda.synchronize()
    mids = layer.intermediates(wl.T)
    sb = to_np(inp.select_bias) if inp.select_bias is not None else None
    ids_o, w_o = oracle_route_from_logits(oracle_logits(inp), wl, sb)
    assert np.array_equal(to_np(mids["topk_ids"]), ids_o)
    toks = sample_tokens(ids_o, n_sample, seed=wl.seed)
    ref = O.moe_loop(to_np(inp.x[torch.as_tensor(toks, device=DEV)]), ids_o[toks], w_o[toks],
                     LazyFp8Experts(c13, s13, True), LazyFp8Experts(c2, s2, False))
    got = to_np(out[torch.as_tensor(toks, device=DEV)])
    assert_close(got, ref, wl.dtype)
    assert torch.isfinite(out.float()).all()


B_CASES = [mi.MIXTRAL, mi.QWEN3, mi.DSV3, mi.GPTOSS.with_T(128)]


@pytest.mark.parametrize("wl", B_CASES, ids=[w.name for w in B_CASES])
def test_version_b_agrees_with_version_a_at_full_size(L, wl):
    """The oracle's two independent forms ("Mixture-of-Experts Kernels: Routing,
    Permutation, and Grouped GEMM", §3: a per-expert loop and a dense run-every-expert
    version that must agree) on a fixed 64-token subset of the full-size layer, tokens of
    the hottest and of the least-loaded non-empty expert among them, with the layer's
    bf16 weights widened exactly: A and B agree to 1e-12 relative (in float64 they differ
    only in the order of the sum over experts). The layer's own output on those tokens is
    then checked against B within the bf16 tolerance."""
    from routing_grouped_gemm_router_gb300.layer import MoELayer
    inp = mi.make_layer(wl, DEV)
    enforce_margins(inp)
    sb = to_np(inp.select_bias) if inp.select_bias is not None else None
    ids, w = oracle_route_from_logits(oracle_logits(inp), wl, sb)
    toks = sample_tokens(ids, 64, seed=wl.seed + 1)
    assert toks.size == 64
    xs = to_np(inp.x[torch.as_tensor(toks, device=DEV)])
    W13, W2 = LazyExpertsF64(inp.W13), LazyExpertsF64(inp.W2)
    a = O.moe_loop(xs, ids[toks], w[toks], W13, W2)
    b = O.moe_dense(xs, ids[toks], w[toks], W13, W2)
    assert np.abs(a - b).max() <= 1e-12 * np.abs(a).max()
    layer = MoELayer(inp.Wg, inp.W13, inp.W2, wl.k, wl.mode, wl.renormalize, wl.scale,
                     wl.n_group, wl.topk_group, inp.logit_bias, inp.select_bias)
    out = layer(inp.x)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(layer.intermediates(wl.T)["topk_ids"]), ids)
    assert_close(to_np(out[torch.as_tensor(toks, device=DEV)]), b, wl.dtype)
