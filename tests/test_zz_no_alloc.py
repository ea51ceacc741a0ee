"""moe_align_noalloc: the align step for callers that cannot give the library scratch memory.

Such callers (an application or server whose device memory belongs to its own pool, or a
path where a cudaMalloc and the device synchronisation it may bring are not allowed) pass only
inputs and outputs; the per-chunk histograms live in a fixed array inside the library. This
test calls the entry point through the C ABI twice in a row on different problems and checks
each result against moe_align given a caller-allocated workspace (integer tables: bit-exact).
It sits in a file of its own, collected last.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    from routing_grouped_gemm_router_gb300 import _lib
    return _lib


def _tables(L, T, k, E, B):
    mp = L.moe_max_padded_rows(T, k, E, B)
    return (torch.full((mp,), -5, dtype=torch.int32, device=DEV),
            torch.full((mp // B,), -5, dtype=torch.int32, device=DEV),
            torch.zeros(1, dtype=torch.int32, device=DEV),
            torch.zeros(E, dtype=torch.int32, device=DEV))


def _with_workspace(L, ids, T, k, E, B):
    sid, eid, npp, cnt = _tables(L, T, k, E, B)
    wsb = L.moe_align_workspace_size(T, k, E, B)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=DEV)
    L.moe_align(ids, T, k, E, B, sid, eid, npp, cnt, ws, wsb)
    return sid, eid, npp, cnt


def _without_workspace(L, ids, T, k, E, B):
    sid, eid, npp, cnt = _tables(L, T, k, E, B)
    L.moe_align_noalloc(ids, T, k, E, B, sid, eid, npp, cnt)
    return sid, eid, npp, cnt


# Two calls in a row that both use the fixed array (T*k > 4096), different shapes and loads,
# then one small problem (one-CTA path).
CALLS = [(8192, 8, 128, 128, 1.0), (3000, 4, 64, 16, 0.0), (100, 2, 8, 16, 0.0)]


def test_noalloc_matches_workspace_align_on_consecutive_calls(L):
    for T, k, E, B, skew in CALLS:
        ids = mi.random_topk_ids(T, k, E, seed=T + E, skew=skew).to(DEV)
        ref = _with_workspace(L, ids, T, k, E, B)
        got = _without_workspace(L, ids, T, k, E, B)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b), f"T={T} k={k} E={E} B={B}"
        n = T * k
        s = got[0].cpu().numpy()
        assert sorted(s[s < n].tolist()) == list(range(n))


def test_noalloc_at_exactly_its_limit(L):
    """The largest accepted problem fills the fixed array to the last int: 524288 rows are
    512 chunks of 1024, times 128 experts = 65536 histogram entries."""
    T, k, E, B = 65536, 8, 128, 128
    assert L.moe_align_workspace_size(T, k, E, B) == 4 * 65536
    ids = mi.random_topk_ids(T, k, E, seed=5, skew=0.5).to(DEV)
    for _ in range(2):
        ref = _with_workspace(L, ids, T, k, E, B)
        got = _without_workspace(L, ids, T, k, E, B)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
    assert L.moe_device_status(True) == 0


def test_noalloc_rejects_problems_beyond_its_fixed_scratch(L):
    # one chunk more than the array holds: 524296 rows are 513 chunks x 128 > 65536 ints
    for T, k, E, B in [(65537, 8, 128, 128), (1 << 17, 8, 128, 128)]:
        with pytest.raises(L.MoeError) as ei:
            L.moe_align_noalloc(16, T, k, E, B, 16, 16, 16)
        assert ei.value.status == L.MOE_ERR_UNSUPPORTED
    assert L.moe_device_status(True) == 0
