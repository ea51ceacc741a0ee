"""Shared test helpers: tolerances, tensor conversion, margin-respecting inputs."""
from __future__ import annotations

import numpy as np
import torch

import moe_inputs as mi
import oracle as O

# Tolerances of the layer output against the float64 oracle.
#  bf16: max|err| <= 1e-2 * max|ref| and relative Frobenius error <= 5e-3;
#  fp32: both <= 1e-5 (tensor-core tf32 could not meet this, so fp32 runs on FFMA).
TOL = {"bf16": (1e-2, 5e-3), "f32": (1e-5, 1e-5)}
MARGIN = 1e-4          # minimum gap between adjacent selection keys in parity inputs
TOPK_W_RTOL = 2e-5     # router weights: fp32 exp/divide vs float64


def to_np(t: torch.Tensor) -> np.ndarray:
    """Exact conversion to float64 (bf16 and fp32 both embed in float64)."""
    return t.detach().float().cpu().double().numpy() if t.is_floating_point() \
        else t.detach().cpu().numpy().astype(np.int64)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bits (uint16) of a bf16 tensor, on the host, without widening it."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def weights_for_oracle(t: torch.Tensor) -> np.ndarray:
    return bf16_bits(t) if t.dtype == torch.bfloat16 else to_np(t)


def err_stats(got: np.ndarray, ref: np.ndarray):
    d = got - ref
    max_rel = np.abs(d).max() / max(np.abs(ref).max(), 1e-300)
    fro = np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-300)
    return max_rel, fro


def assert_close(got, ref, dtype: str, what: str = "out"):
    tmax, tfro = TOL[dtype]
    max_rel, fro = err_stats(np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64))
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert max_rel <= tmax and fro <= tfro, \
        f"{what}: max|err|/max|ref| = {max_rel:.3e} (tol {tmax}), rel Frobenius = {fro:.3e} (tol {tfro})"
    return max_rel, fro


def oracle_logits(inp: mi.LayerInputs) -> np.ndarray:
    lb = to_np(inp.logit_bias) if inp.logit_bias is not None else None
    return O.router_logits(to_np(inp.x), to_np(inp.Wg), lb if inp.wl.mode == 0 else None)


def oracle_route_from_logits(logits: np.ndarray, wl: mi.Workload, select_bias=None):
    return O.route(logits, wl.k, wl.mode, wl.renormalize, wl.scale, wl.n_group, wl.topk_group,
                   select_bias)


def enforce_margins(inp: mi.LayerInputs, margin: float = MARGIN, max_rounds: int = 20) -> int:
    """Redraw token rows whose top-k selection keys (float64, from the stored inputs) have an
    adjacent gap <= margin. Returns the number of redraws."""
    wl = inp.wl
    sb = to_np(inp.select_bias) if inp.select_bias is not None else None
    Wg = to_np(inp.Wg)
    lb = to_np(inp.logit_bias) if (inp.logit_bias is not None and wl.mode == 0) else None
    redraws = 0
    rows = np.arange(wl.T)
    for attempt in range(max_rounds):
        xs = to_np(inp.x[torch.as_tensor(rows, device=inp.x.device)])
        l = O.router_logits(xs, Wg, lb)
        m = O.selection_margins(l, wl.k, wl.mode, wl.n_group, wl.topk_group, sb)
        bad = rows[m <= margin]
        if bad.size == 0:
            return redraws
        redraws += bad.size
        mi.redraw_rows(inp.x, bad.tolist(), wl.seed, attempt)
        rows = bad
    raise RuntimeError("could not reach the routing margin")


class LazyExperts:
    """Expert weights left on the device; ``[e]`` copies one expert's bf16 bits (or fp32
    values) to the host on demand, so the oracle never holds a multi-GB copy."""

    def __init__(self, W: torch.Tensor):
        self.W = W
        self.shape = tuple(W.shape)

    def __getitem__(self, e):
        return weights_for_oracle(self.W[int(e)])


class LazyExpertsF64:
    """As LazyExperts, but each expert is widened to float64 on the device (exact for bf16
    and fp32) before it is copied: for the tests that walk every expert of a multi-GB layer
    several times, where widening on the host would dominate."""

    def __init__(self, W: torch.Tensor):
        self.W = W
        self.shape = tuple(W.shape)

    def __getitem__(self, e):
        return self.W[int(e)].double().cpu().numpy()


class LazyFp8Experts:
    """FP8 expert weights (codes + block scales) left on the device; ``[e]`` dequantises one
    expert on the host with the oracle (code * scale of its 128 x 128 block)."""

    def __init__(self, codes: torch.Tensor, scales: torch.Tensor, w13: bool):
        self.codes, self.scales, self.w13 = codes, scales, w13
        self.shape = tuple(codes.shape)

    def __getitem__(self, e):
        c = self.codes[int(e)].cpu().numpy()[None]
        s = self.scales[int(e)].double().cpu().numpy()[None]
        return (O.dequant_w13(c, s) if self.w13 else O.dequant_blockwise(c, s))[0]


def sample_tokens(ids: np.ndarray, n: int, seed: int = 0) -> np.ndarray:
    """n token indices: tokens routed to the hottest expert and to the least-loaded
    non-empty expert, then uniform picks."""
    E = int(ids.max()) + 1
    counts = np.bincount(ids.ravel(), minlength=E)
    hot = int(np.argmax(counts))
    nz = np.nonzero(counts)[0]
    cold = int(nz[np.argmin(counts[nz])])
    pick = []
    for e in (hot, cold):
        pick += np.nonzero((ids == e).any(1))[0][:max(1, n // 8)].tolist()
    rng = np.random.default_rng(seed)
    rest = rng.permutation(ids.shape[0])
    for t in rest:
        if len(set(pick)) >= n:
            break
        pick.append(int(t))
    return np.array(sorted(set(pick)))[:max(n, 1)]
