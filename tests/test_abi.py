"""The C-ABI library loads, exports every declared entry point, and its host-side logic
(argument checks, sizes, workspace layout) behaves, all without a GPU."""
import ctypes
import os
import re

import pytest
import torch

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from conftest import build_library
    build_library()
    from routing_grouped_gemm_router_gb300 import _lib
    return _lib


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(moe_\w+)\s*\(", src)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(L):
    decl = _declared()
    assert "moe_forward" in decl and "moe_align" in decl and "moe_route" in decl
    cdll = ctypes.CDLL(L.LIB_PATH)
    missing = [n for n in decl if not hasattr(cdll, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert set(decl) <= set(L.EXPORTED) | set(decl)
    assert L.moe_abi_version() == 9


def test_status_strings(L):
    for s in range(5):
        assert L.status_string(s)


@pytest.mark.parametrize("T,k,E,B", [(64, 2, 8, 16), (1, 4, 128, 128), (4096, 8, 256, 128),
                                     (3, 3, 5, 4), (37, 1, 8, 16)])
def test_max_padded_matches_oracle(L, T, k, E, B):
    assert L.moe_max_padded_rows(T, k, E, B) == O.max_padded_rows(T, k, E, B)


def test_block_m_and_workspace(L):
    cfg = L.make_config(4096, 4096, 14336, 8, 2, L.MOE_BF16)
    assert L.moe_block_m(cfg) == 128
    lay = L.moe_workspace_layout(cfg)
    assert lay.block_m == 128 and lay.max_padded == O.max_padded_rows(4096, 2, 8, 128)
    offs = [lay.logits, lay.topk_ids, lay.topk_w, lay.sorted_ids, lay.expert_ids,
            lay.num_post_padded, lay.counts, lay.align_scratch, lay.act, lay.y]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    assert lay.total >= lay.y + 4096 * 2 * 4096 * 2
    assert L.moe_workspace_size(cfg) == lay.total
    cfg32 = L.make_config(64, 64, 96, 8, 2, L.MOE_F32)
    assert L.moe_block_m(cfg32) == 16


def test_small_batch_predicate(L):
    """bf16 layers of at most 2 tokens (24 with FP8 weights) take the small-batch grouped
    GEMMs; fp32 layers, larger batches and bad configurations do not (host arithmetic)."""
    assert L.moe_small_batch(L.make_config(1, 2880, 2880, 128, 4, L.MOE_BF16))
    assert L.moe_small_batch(L.make_config(2, 7168, 2048, 256, 8, L.MOE_BF16))
    assert not L.moe_small_batch(L.make_config(3, 2880, 2880, 128, 4, L.MOE_BF16))
    assert not L.moe_small_batch(L.make_config(4, 64, 96, 8, 2, L.MOE_F32))
    assert not L.moe_small_batch(L.make_config(0, 64, 96, 8, 2, L.MOE_BF16))
    s13, s2 = torch.ones(128, 2, 23, 23), torch.ones(128, 23, 23)  # scale grids (host only)
    fp8 = lambda T: L.make_config(T, 2880, 2880, 128, 4, L.MOE_BF16, w13_scale=s13,  # noqa: E731
                                  w2_scale=s2)
    assert L.moe_small_batch(fp8(24)) and not L.moe_small_batch(fp8(25))


def test_gemm_kernel_query(L):
    """moe_gemm_kernel names the grouped-GEMM kernels each configuration runs: fp32 layers the
    CUDA-core tiles, bf16 layers by batch size (2 tokens, 24 with FP8 weights, 128), shared
    experts counted into the effective top-k, and 0 for a bad configuration (host only)."""
    mk = lambda T, **kw: L.make_config(T, 2880, 2880, 128, 4, L.MOE_BF16, **kw)  # noqa: E731
    assert L.moe_gemm_kernel(L.make_config(4, 64, 96, 8, 2, L.MOE_F32)) == L.MOE_GEMM_SIMT
    assert L.moe_gemm_kernel(mk(1)) == L.MOE_GEMM_SMALL_BATCH
    assert L.moe_gemm_kernel(mk(2)) == L.MOE_GEMM_SMALL_BATCH
    assert L.moe_gemm_kernel(mk(3)) == L.MOE_GEMM_DECODE_TC
    assert L.moe_gemm_kernel(mk(128)) == L.MOE_GEMM_DECODE_TC
    assert L.moe_gemm_kernel(mk(129)) == L.MOE_GEMM_PAIR_TC
    assert L.moe_gemm_kernel(mk(16384)) == L.MOE_GEMM_PAIR_TC
    s13, s2 = torch.ones(128, 2, 23, 23), torch.ones(128, 23, 23)  # scale grids (host only)
    assert L.moe_gemm_kernel(mk(24, w13_scale=s13, w2_scale=s2)) == L.MOE_GEMM_SMALL_BATCH
    assert L.moe_gemm_kernel(mk(25, w13_scale=s13, w2_scale=s2)) == L.MOE_GEMM_DECODE_TC
    assert L.moe_gemm_kernel(mk(0)) == L.MOE_GEMM_INVALID
    for T in (1, 2, 3, 12, 13, 128, 129, 4096):
        assert L.moe_small_batch(mk(T)) == (L.moe_gemm_kernel(mk(T)) == L.MOE_GEMM_SMALL_BATCH)


def test_fp8_prefill_workspace_holds_bf16_weights(L):
    """With FP8 weights, the batches the CTA-pair kernels take with at least 256 routed rows
    per expert convert each grouped GEMM's weights to bf16 in the workspace first: its GEMM
    scratch region holds E slots (shared experts included) of 2I x H bf16 weights; other
    batches and bf16 weights need none."""
    E, H, I, ns = 8, 512, 384, 1
    s13, s2 = torch.ones(E + ns, 2, 3, 4), torch.ones(E + ns, 4, 3)  # scale grids (host only)
    fp8 = lambda T: L.make_config(T, H, I, E, 2, L.MOE_BF16, n_shared=ns,  # noqa: E731
                                  w13_scale=s13, w2_scale=s2)
    lay = L.moe_workspace_layout(fp8(1024))
    assert lay.total - lay.gemm_scratch >= (E + ns) * 2 * I * H * 2
    few = L.make_config(512, H, I, 64, 2, L.MOE_BF16, w13_scale=torch.ones(64, 2, 3, 4),
                        w2_scale=torch.ones(64, 4, 3))  # 16 rows an expert: converted in-GEMM
    for cfg in (fp8(64), few, L.make_config(1024, H, I, E, 2, L.MOE_BF16, n_shared=ns)):
        lay = L.moe_workspace_layout(cfg)
        assert lay.total == lay.gemm_scratch


def test_decode_parity_cases_take_their_paths(L):
    """The decode layers of the GPU parity tests exercise the paths they are named for: the
    9-token layer and the FP8 layers of 25 tokens and more run the decode tensor-core GEMMs,
    the 1- and 2-token layers and the 24-token FP8 layer the small-batch kernels."""
    dec = L.MOE_GEMM_DECODE_TC
    assert L.moe_gemm_kernel(L.make_config(9, 320, 448, 8, 4, L.MOE_BF16)) == dec
    s13, s2 = torch.ones(8, 2, 3, 3), torch.ones(8, 3, 3)  # scale grids (host only)
    fp8 = lambda T: L.make_config(T, 320, 272, 8, 2, L.MOE_BF16, w13_scale=s13,  # noqa: E731
                                  w2_scale=s2)
    assert L.moe_gemm_kernel(fp8(24)) == L.MOE_GEMM_SMALL_BATCH
    for T in (28, 64):
        assert L.moe_gemm_kernel(fp8(T)) == dec
    for T, H, I, E, k in ((1, 2880, 2880, 128, 4), (2, 2880, 2880, 32, 4), (2, 1000, 776, 4, 2)):
        assert L.moe_small_batch(L.make_config(T, H, I, E, k, L.MOE_BF16))


@pytest.mark.parametrize("kw", [dict(T=0), dict(k=9), dict(H=12), dict(I=100), dict(E=0)])
def test_invalid_configs_rejected(L, kw):
    a = dict(T=4, H=64, I=96, E=8, k=2)
    a.update(kw)
    cfg = L.make_config(a["T"], a["H"], a["I"], a["E"], a["k"], L.MOE_F32)
    with pytest.raises(L.MoeError) as ei:
        L.moe_workspace_size(cfg)
    assert ei.value.status == L.MOE_ERR_INVALID_ARG


def test_grouped_router_config_checks(L):
    bad_group = L.make_config(4, 64, 96, 10, 2, L.MOE_BF16, L.MOE_ROUTE_SIGMOID_GROUPED,
                              n_group=4, topk_group=2)
    with pytest.raises(L.MoeError):
        L.moe_workspace_size(bad_group)
    too_few = L.make_config(4, 64, 96, 16, 8, L.MOE_BF16, L.MOE_ROUTE_SIGMOID_GROUPED,
                            n_group=8, topk_group=2)   # 2 groups x 2 experts < k = 8
    with pytest.raises(L.MoeError):
        L.moe_workspace_size(too_few)
    too_many_e = L.make_config(4, 64, 96, 1024, 2, L.MOE_BF16)
    with pytest.raises(L.MoeError) as ei:
        L.moe_workspace_size(too_many_e)
    assert ei.value.status == L.MOE_ERR_UNSUPPORTED


def test_null_pointers_rejected_before_any_launch(L):
    cfg = L.make_config(4, 64, 96, 8, 2, L.MOE_F32)
    with pytest.raises(L.MoeError) as ei:
        L.moe_route(cfg, 0, 0, 0, 0, 0, stream=0)
    assert ei.value.status == L.MOE_ERR_INVALID_ARG
    with pytest.raises(L.MoeError) as ei:
        L.moe_forward(cfg, 16, 16, 16, 16, 16, 0, 0, stream=0)
    assert ei.value.status == L.MOE_ERR_WORKSPACE
    with pytest.raises(L.MoeError) as ei:
        L.moe_align(0, 4, 2, 8, 16, 0, 0, 0, stream=0)
    assert ei.value.status == L.MOE_ERR_INVALID_ARG


def test_align_workspace_sizes(L):
    assert L.moe_align_workspace_size(64, 2, 8, 16) == 0           # one-CTA path
    assert L.moe_align_workspace_size(8192, 8, 128, 128) >= 64 * 128 * 4
    with pytest.raises(L.MoeError) as ei:
        L.moe_align(16, 8192, 8, 128, 128, 16, 16, 16, ws=None, ws_bytes=0, stream=0)
    assert ei.value.status == L.MOE_ERR_WORKSPACE


def test_fp8_weight_config_checks(L):
    ok = L.make_config(4, 64, 96, 8, 2, L.MOE_BF16, w13_scale=256, w2_scale=512)
    assert ok.weight_format == L.MOE_WEIGHTS_FP8_E4M3_B128
    assert L.moe_workspace_size(ok) > 0
    cases = [(L.make_config(4, 64, 96, 8, 2, L.MOE_F32, w13_scale=256, w2_scale=512),
              L.MOE_ERR_UNSUPPORTED),                                   # fp32 activations
             (L.make_config(4, 72, 96, 8, 2, L.MOE_BF16, w13_scale=256, w2_scale=512),
              L.MOE_ERR_INVALID_ARG),                                   # H % 16
             (L.make_config(4, 64, 104, 8, 2, L.MOE_BF16, w13_scale=256, w2_scale=512),
              L.MOE_ERR_INVALID_ARG),                                   # I % 16
             (L.make_config(4, 64, 96, 8, 2, L.MOE_BF16, w13_scale=256),
              L.MOE_ERR_INVALID_ARG),                                   # a scale missing
             (L.make_config(4, 64, 96, 8, 2, L.MOE_BF16, w13_scale=258, w2_scale=512),
              L.MOE_ERR_INVALID_ARG)]                                   # misaligned scale
    for cfg, want in cases:
        with pytest.raises(L.MoeError) as ei:
            L.moe_workspace_size(cfg)
        assert ei.value.status == want
