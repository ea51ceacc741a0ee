"""Seeded synthetic inputs for the fused MoE feed-forward layer.

This module only draws random numbers and lays them out; it holds none of the
layer's arithmetic (no routing, no top-k, no GEMM). Both the CUDA path's tests
and the float64 oracle take their inputs from here.

Workloads follow the model table of "Mixture-of-Experts Kernels: Routing,
Permutation, and Grouped GEMM", §1 (Mixtral-8x7B, gpt-oss-120b, Qwen3-235B-A22B,
DeepSeek-V3), with the initialisation of that page's §3 ``make_layer``:
router and gate/up projections ~ N(0, 1/H), down projection ~ N(0, 1/I), tokens
~ N(0, 1). Weights use the nn.Linear ``[E, N, K]`` layout: ``W13[E, 2I, H]`` holds
the gate projection W1 in rows ``0..I-1`` and the up projection W3 in rows
``I..2I-1`` of each expert; ``W2[E, H, I]``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

# Routing modes (same numbering as the C header).
ROUTE_SOFTMAX = 0
ROUTE_SIGMOID_GROUPED = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    """One layer shape plus its router settings and input distribution."""

    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    dtype: str  # "f32" or "bf16"
    mode: int = ROUTE_SOFTMAX
    renormalize: bool = True
    scale: float = 1.0
    n_group: int = 1
    topk_group: int = 1
    logit_bias_std: float = 0.0   # mode 0: per-expert offset added to the logits
    select_bias_std: float = 0.0  # mode 1: selection-only bias
    seed: int = 0

    def with_T(self, T: int) -> "Workload":
        return dataclasses.replace(self, T=T, name=f"{self.name.split('@')[0]}@T={T}")

    def small(self, T: int, H: int, I: int) -> "Workload":
        """Same router/expert structure at a reduced size (for fast parity)."""
        return dataclasses.replace(self, T=T, H=H, I=I, name=f"{self.name}-small")

    @property
    def flops(self) -> int:
        """Useful expert FLOPs: 6*T*k*H*I (two GEMMs, padding and router excluded)."""
        return 6 * self.T * self.k * self.H * self.I


# The five workloads: the page's tiny fp32 layer, then four bf16 layers shaped like the
# §1 model table. The gpt-oss decode entry is swept over T in {1, 8, 32, 128}.
TINY_F32 = Workload("tiny-f32", T=64, H=64, I=96, E=8, k=2, dtype="f32", seed=0)
MIXTRAL = Workload("mixtral-prefill", T=4096, H=4096, I=14336, E=8, k=2, dtype="bf16", seed=1)
QWEN3 = Workload("qwen3-skewed", T=8192, H=4096, I=1536, E=128, k=8, dtype="bf16",
                 logit_bias_std=1.5, seed=2)
DSV3 = Workload("deepseek-v3", T=4096, H=7168, I=2048, E=256, k=8, dtype="bf16",
                mode=ROUTE_SIGMOID_GROUPED, scale=2.5, n_group=8, topk_group=4,
                select_bias_std=0.05, seed=3)
GPTOSS = Workload("gpt-oss-decode", T=128, H=2880, I=2880, E=128, k=4, dtype="bf16", seed=4)
GPTOSS_T = (1, 8, 32, 128)

WORKLOADS = {w.name: w for w in (TINY_F32, MIXTRAL, QWEN3, DSV3, GPTOSS)}


@dataclasses.dataclass
class LayerInputs:
    """Tensors of one layer instance (all on one device)."""

    wl: Workload
    x: torch.Tensor            # [T, H]
    Wg: torch.Tensor           # [E, H]
    W13: torch.Tensor          # [E, 2I, H]
    W2: torch.Tensor           # [E, H, I]
    logit_bias: Optional[torch.Tensor] = None   # [E] fp32 (mode 0)
    select_bias: Optional[torch.Tensor] = None  # [E] fp32 (mode 1)


def _dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_cast(shape, std: float, g: torch.Generator, device, dtype, chunk_rows: int = 1):
    """N(0, std^2) drawn in fp32 slab by slab (dim 0) and cast to ``dtype``.

    Drawing per slab keeps the fp32 staging buffer small for multi-GB weights.
    """
    out = torch.empty(shape, dtype=dtype, device=device)
    for i in range(0, shape[0], chunk_rows):
        sl = out[i:i + chunk_rows]
        sl.copy_(torch.randn(sl.shape, generator=g, device=device, dtype=torch.float32) * std)
    return out


def make_layer(wl: Workload, device="cpu", seed: Optional[int] = None) -> LayerInputs:
    """Draw one layer instance of workload ``wl`` on ``device``.

    The same (workload, device type, seed) always gives the same tensors. The CUDA
    and CPU generators differ, so big layers are drawn on the GPU and copied to the
    host for the oracle.
    """
    seed = wl.seed if seed is None else seed
    dt = _dtype(wl.dtype)
    g = _gen(device, seed)
    T, H, I, E = wl.T, wl.H, wl.I, wl.E
    x = _randn_cast((T, H), 1.0, g, device, dt, chunk_rows=max(1, T))
    Wg = _randn_cast((E, H), 1.0 / math.sqrt(H), g, device, dt, chunk_rows=E)
    W13 = _randn_cast((E, 2 * I, H), 1.0 / math.sqrt(H), g, device, dt)
    W2 = _randn_cast((E, H, I), 1.0 / math.sqrt(I), g, device, dt)
    lb = sb = None
    if wl.logit_bias_std > 0:
        lb = torch.randn(E, generator=g, device=device, dtype=torch.float32) * wl.logit_bias_std
    if wl.select_bias_std > 0:
        sb = torch.randn(E, generator=g, device=device, dtype=torch.float32) * wl.select_bias_std
    return LayerInputs(wl, x, Wg, W13, W2, lb, sb)


def quantize_fp8_blocks(W: torch.Tensor, block: int = 128):
    """FP8 E4M3 codes (uint8) and fp32 scales of W[E, N, K], one scale per block x block
    tile: the smallest power of two with amax / scale <= 448 (the E4M3 maximum), so that
    code * scale reproduces W to E4M3 precision. Input preparation only: the layer takes the
    codes and scales as they are, and so does the oracle."""
    E, N, K = W.shape
    RB, KB = -(-N // block), -(-K // block)
    codes = torch.empty((E, N, K), dtype=torch.uint8, device=W.device)
    scales = torch.empty((E, RB, KB), dtype=torch.float32, device=W.device)
    for e in range(E):
        w = torch.zeros(RB * block, KB * block, dtype=torch.float32, device=W.device)
        w[:N, :K] = W[e].float()
        amax = w.view(RB, block, KB, block).abs().amax(dim=(1, 3)) / 448.0
        m, ex = torch.frexp(amax.clamp_min(2.0 ** -100))   # amax = m * 2^ex, m in [0.5, 1)
        sc = torch.ldexp(torch.ones_like(m), ex - (m == 0.5).to(ex.dtype))
        q = w / sc.repeat_interleave(block, 0).repeat_interleave(block, 1)
        codes[e] = q[:N, :K].to(torch.float8_e4m3fn).view(torch.uint8)
        scales[e] = sc
    return codes, scales


def quantize_fp8_w13(W13: torch.Tensor, block: int = 128):
    """Codes of W13[E, 2I, H] and scales[E, 2, ceil(I/block), ceil(H/block)]: the gate rows
    and the up rows are quantised as two separate matrices."""
    I = W13.shape[1] // 2
    cg, sg = quantize_fp8_blocks(W13[:, :I], block)
    cu, su = quantize_fp8_blocks(W13[:, I:], block)
    return torch.cat([cg, cu], 1), torch.stack([sg, su], 1)


def redraw_rows(x: torch.Tensor, rows, seed: int, attempt: int) -> None:
    """Replace token rows ``rows`` of ``x`` in place by fresh N(0,1) draws.

    Row t on attempt a is drawn from a CPU generator seeded by (seed, t, a), so the
    redraw is the same on every machine and independent of the device ``x`` is on.
    """
    for t in rows:
        g = _gen("cpu", (seed * 1_000_003 + int(t) * 7919 + attempt * 104_729) % (2**63 - 1))
        r = torch.randn(x.shape[1], generator=g, dtype=torch.float32)
        x[int(t)].copy_(r.to(x.dtype))


# ---------------------------------------------------------------------------------------
# The pages' own seeded examples (reproduced draw for draw, fp32).
# ---------------------------------------------------------------------------------------

def page_tiny_layer():
    """The §3 ground-truth script of the routing/grouped-GEMM page.

    ``torch.manual_seed(0)``; ``x = randn(64, 64)``; then ``make_layer(64, 96, 8, seed=0)``
    draws the router, W1, W3 (scaled 1/sqrt(H)) and W2 (scaled 1/sqrt(I)) from its own
    generator. Returns fp32 ``x, Wg, W1, W3, W2`` on the CPU.
    """
    T, H, I, E = 64, 64, 96, 8
    torch.manual_seed(0)
    x = torch.randn(T, H)
    return (x,) + _page_make_layer(H, I, E, seed=0)


def _page_make_layer(H, I, E, seed):
    g = torch.Generator().manual_seed(seed)
    s = 1.0 / H ** 0.5
    wg = torch.randn(E, H, generator=g) * s
    w1 = torch.randn(E, I, H, generator=g) * s
    w3 = torch.randn(E, I, H, generator=g) * s
    w2 = torch.randn(E, H, I, generator=g) / I ** 0.5
    return wg, w1, w3, w2


# §6 test matrix of the same page: (name, tokens, experts, top_k, bias toward expert 0).
PAGE_FUSED_CASES = (
    ("uniform E=8 k=2", 64, 8, 2, 0.0),
    ("skewed E=16 k=4", 50, 16, 4, 3.0),
    ("decode T=1 k=2", 1, 8, 2, 0.0),
    ("top-1 E=8 k=1", 37, 8, 1, 0.0),
)


def page_fused_case(T, E, bias, H=64, I=96):
    """One §6 test case: seed 1 for tokens, ``make_layer(H, I, E, seed=2)`` for weights,
    and a unit direction ``u`` that raises expert 0's logit when ``bias`` > 0.
    Returns fp32 ``x, Wg, W1, W3, W2``."""
    torch.manual_seed(1)
    wg, w1, w3, w2 = _page_make_layer(H, I, E, seed=2)
    u = torch.nn.functional.normalize(torch.randn(H), dim=0)
    wg[0] += bias * u
    x = torch.randn(T, H) + 1.5 * u
    return x, wg, w1, w3, w2


def page_deepseek_toy():
    """§4 router example: ``torch.manual_seed(0)``; logits ``randn(4, 16)``; a bias of 0.5
    on experts 0, 4, 8, 12. Returns fp32 ``logits [4,16]`` and ``bias [16]``."""
    torch.manual_seed(0)
    logits = torch.randn(4, 16)
    bias = torch.zeros(16)
    bias[torch.arange(16) % 4 == 0] = 0.5
    return logits, bias


def page_align_example():
    """§5 worked example (the one from vLLM's moe_align_block_size docstring):
    topk_ids for 4 tokens, k=3, E=5, BLOCK_M=4."""
    return torch.tensor([[2, 3, 4], [1, 2, 4], [1, 3, 4], [1, 2, 3]], dtype=torch.int32)


def random_topk_ids(T, k, E, seed, skew=0.0):
    """Distinct-per-row expert ids (for align tests), optionally Zipf-skewed."""
    g = _gen("cpu", seed)
    p = 1.0 / torch.arange(1, E + 1, dtype=torch.float64) ** skew
    p = (p / p.sum()).expand(T, E)
    return torch.multinomial(p, k, replacement=False, generator=g).to(torch.int32)
