"""Float64 CPU oracle for the fused Mixture-of-Experts feed-forward layer.

TEST INFRASTRUCTURE ONLY. This module is the plain, slow, obviously correct statement
of what the layer computes. Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import it; the product path never calls it and
shares no code with the CUDA library.

Sources (page title and section):
  [P2] "Mixture-of-Experts Kernels: Routing, Permutation, and Grouped GEMM"
       §1 (layer definition and model table), §2 (route -> align -> grouped GEMM ->
       combine, flat row r = t*k + j), §3 (ground truth: per-expert loop and dense
       run-every-expert version), §4 (DeepSeek-style grouped sigmoid router), §5 (the
       sorted_ids / expert_ids indirection table), §6 (gathered GEMM1, SwiGLU,
       GEMM2 with the router weight, sum over k).
  [P3] "fused-moe-kernel" skill card: Token-Expert Routing, Common Pitfalls.

Everything is float64 (inputs given in fp32/bf16 convert exactly). Readings where the
pages are silent:
  * top-k order: larger key first; an exact tie goes to the lower expert (or group) id;
  * slots j of a token are in that descending key order (mode 1: the biased key);
  * rows inside one expert's run of sorted_ids are in ascending flat row r (stable);
  * padding rows and the unused tail of sorted_ids hold the sentinel T*k; unused
    tail entries of expert_ids hold -1;
  * combine sums slots j = 0..k-1 in order.

Parity status: every function here is pinned by tests against values the pages print,
brute force on tiny inputs, closed forms and invariants (see tests/test_oracle_pins.py).
"""
from __future__ import annotations

import itertools
from typing import Optional, Tuple

import numpy as np

SOFTMAX = 0
SIGMOID_GROUPED = 1


# ----------------------------------------------------------------------------- inputs

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact bf16 -> float64: a bf16 is the top 16 bits of an IEEE float32."""
    u32 = bits.astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Decode FP8 E4M3 (OCP "FN" variant) bytes from the format's definition: 1 sign bit,
    4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); the
    all-ones code S.1111.111 is NaN (no infinities), so the largest finite value is 448."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return sign * val


def dequant_blockwise(codes: np.ndarray, scales: np.ndarray, block: int = 128) -> np.ndarray:
    """FP8 expert weights with their scales ([P2] §8: one byte per weight; §9: the FP8 weight
    variants of the fused kernel; §10: FP8 scale handling checked against a wide reference):
    w[..., n, c] = e4m3(codes[..., n, c]) * scales[..., n // block, c // block].
    Reading: the pages name FP8 scales but not their granularity; one scale per
    block x block tile of each expert matrix (block = 128) is the plainest form that
    covers per-expert scales (one tile) as a special case."""
    v = e4m3_to_f64(codes)
    sc = f64(scales)
    n, k = v.shape[-2], v.shape[-1]
    rows = np.arange(n) // block
    cols = np.arange(k) // block
    return v * sc[..., rows[:, None], cols[None, :]]


def dequant_w13(codes13: np.ndarray, scales13: np.ndarray, block: int = 128) -> np.ndarray:
    """FP8 W13[E, 2I, H]: the gate rows 0..I-1 and the up rows I..2I-1 are two matrices,
    each with its own block grid (scales13[E, 2, ceil(I/block), ceil(H/block)]), as when
    gate and up projections are quantised separately and then stacked."""
    I = codes13.shape[-2] // 2
    gate = dequant_blockwise(codes13[..., :I, :], scales13[:, 0], block)
    up = dequant_blockwise(codes13[..., I:, :], scales13[:, 1], block)
    return np.concatenate([gate, up], axis=-2)


# ----------------------------------------------------------------------------- top-k

def topk_desc(keys: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries of each row, in descending key order.

    Ties go to the lower index (np.lexsort sorts by the last key first: -key, then index).
    """
    keys = f64(keys)
    n = keys.shape[-1]
    idx = np.broadcast_to(np.arange(n), keys.shape)
    out = np.empty(keys.shape[:-1] + (k,), dtype=np.int64)
    for row in np.ndindex(keys.shape[:-1]):
        order = np.lexsort((idx[row], -keys[row]))
        out[row] = order[:k]
    return out


# ----------------------------------------------------------------------------- routers

def router_logits(x, Wg, logit_bias=None) -> np.ndarray:
    """[P2 §3] logits = x @ Wg^T, plus an optional per-expert offset (Qwen3-shaped skew)."""
    l = f64(x) @ f64(Wg).T
    if logit_bias is not None:
        l = l + f64(logit_bias)[None, :]
    return l


def softmax(l: np.ndarray) -> np.ndarray:
    m = l.max(axis=-1, keepdims=True)
    e = np.exp(l - m)
    return e / e.sum(axis=-1, keepdims=True)


def route_softmax(logits, k: int, renormalize: bool = True) -> Tuple[np.ndarray, np.ndarray]:
    """[P2 §3 route] softmax over the E experts, keep the k largest probabilities,
    optionally renormalise the k kept weights to sum to 1.

    Softmax is monotonic, so the kept experts are the k largest logits.
    Returns ids [T,k] (int64) and weights [T,k] (float64).
    """
    p = softmax(f64(logits))
    ids = topk_desc(p, k)
    w = np.take_along_axis(p, ids, axis=-1)
    if renormalize:
        w = w / w.sum(axis=-1, keepdims=True)
    return ids, w


def route_topk_then_softmax(logits, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """The gpt-oss form ([P2 §1] table: "softmax over top-4"): take the k largest logits,
    then a softmax over just those k. An independent routine; equal to
    ``route_softmax(..., renormalize=True)`` in exact arithmetic."""
    l = f64(logits)
    ids = topk_desc(l, k)
    sel = np.take_along_axis(l, ids, axis=-1)
    e = np.exp(sel - sel[:, :1])
    return ids, e / e.sum(axis=-1, keepdims=True)


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def route_sigmoid_grouped(logits, k: int, n_group: int, topk_group: int,
                          select_bias=None, scale: float = 1.0,
                          renormalize: bool = True) -> Tuple[np.ndarray, np.ndarray]:
    """[P2 §4] DeepSeek-V3 routing.

    s = sigmoid(logits); c = s + bias (the bias steers selection only); each of the
    n_group groups of E/n_group consecutive experts is scored by the sum of its two
    largest c; the topk_group best groups stay eligible; the k largest c among the
    eligible experts are chosen; their weights come from the UNBIASED s, renormalised
    over the k and then multiplied by ``scale`` (routed_scaling_factor).
    """
    l = f64(logits)
    T, E = l.shape
    s = sigmoid(l)
    c = s + (f64(select_bias)[None, :] if select_bias is not None else 0.0)
    per = E // n_group
    grouped = c.reshape(T, n_group, per)
    top2 = min(2, per)
    gscore = np.sort(grouped, axis=-1)[..., ::-1][..., :top2].sum(-1)    # [T, G]
    keep = topk_desc(gscore, topk_group)                                  # [T, topk_group]
    eligible = np.zeros((T, n_group), dtype=bool)
    np.put_along_axis(eligible, keep, True, axis=-1)
    eligible = np.repeat(eligible, per, axis=1)                          # [T, E]
    masked = np.where(eligible, c, -np.inf)
    ids = topk_desc(masked, k)
    w = np.take_along_axis(s, ids, axis=-1)
    if renormalize:
        w = w / w.sum(axis=-1, keepdims=True)
    return ids, scale * w


def route(logits, k, mode=SOFTMAX, renormalize=True, scale=1.0, n_group=1, topk_group=1,
          select_bias=None):
    """Dispatch on the routing mode (0: softmax top-k, 1: grouped sigmoid)."""
    if mode == SOFTMAX:
        ids, w = route_softmax(logits, k, renormalize)
        return ids, w * scale
    return route_sigmoid_grouped(logits, k, n_group, topk_group, select_bias, scale, renormalize)


def selection_margins(logits, k, mode=SOFTMAX, n_group=1, topk_group=1, select_bias=None):
    """Smallest gap, per token, between adjacent keys among the top k+1 selection keys
    (and, in mode 1, between the topk_group-th and next group score). Inputs whose gaps
    all exceed a threshold route the same way under any small perturbation of logits."""
    l = f64(logits)
    T, E = l.shape
    if mode == SOFTMAX:
        keys = l
    else:
        c = sigmoid(l) + (f64(select_bias)[None, :] if select_bias is not None else 0.0)
        per = E // n_group
        gs = np.sort(c.reshape(T, n_group, per), axis=-1)[..., ::-1][..., :min(2, per)].sum(-1)
        gsort = np.sort(gs, axis=-1)[:, ::-1]
        ggap = (gsort[:, topk_group - 1] - gsort[:, topk_group]) if topk_group < n_group \
            else np.full(T, np.inf)
        keep = topk_desc(gs, topk_group)
        elig = np.zeros((T, n_group), dtype=bool)
        np.put_along_axis(elig, keep, True, axis=-1)
        keys = np.where(np.repeat(elig, per, axis=1), c, -np.inf)
    srt = np.sort(keys, axis=-1)[:, ::-1]
    m = min(k + 1, E)
    gaps = srt[:, :m - 1] - srt[:, 1:m]
    gaps = np.where(np.isfinite(gaps), gaps, np.inf)
    out = gaps.min(axis=-1) if m > 1 else np.full(T, np.inf)
    if mode != SOFTMAX:
        out = np.minimum(out, ggap)
    return out


# ----------------------------------------------------------------------------- align

def max_padded_rows(T: int, k: int, E: int, block_m: int) -> int:
    """Worst-case padded length of sorted_ids: every expert that can hold a row pads at
    most block_m-1 slots, and the padded total is a whole number of tiles, so the bound
    T*k + min(E, T*k)*(block_m-1) rounded down to a multiple of block_m also holds."""
    n = T * k
    return (n + min(E, n) * (block_m - 1)) // block_m * block_m


def moe_align(topk_ids, block_m: int, E: int, max_padded: Optional[int] = None):
    """[P2 §5] histogram -> pad each expert's run to a multiple of block_m -> exclusive
    scan -> scatter each flat row r = t*k + j to start[e] + (its rank among e's rows).

    Returns (sorted_ids, expert_ids, total, counts). With ``max_padded`` the arrays have
    fixed length: sorted_ids tail = sentinel T*k, expert_ids tail = -1.
    """
    flat = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    n = flat.size
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:                                   # 1. histogram
        counts[e] += 1
    padded = (counts + block_m - 1) // block_m * block_m   # 2. round up to block_m
    starts = np.zeros(E, dtype=np.int64)             # 3. exclusive scan
    acc = 0
    for e in range(E):
        starts[e] = acc
        acc += padded[e]
    total = int(acc)
    L = total if max_padded is None else max_padded
    sorted_ids = np.full(L, n, dtype=np.int64)       # sentinel = T*k
    fill = starts.copy()
    for r in range(n):                               # 4. scatter, stable in r
        e = flat[r]
        sorted_ids[fill[e]] = r
        fill[e] += 1
    n_tiles = L // block_m if max_padded is not None else total // block_m
    expert_ids = np.full(n_tiles, -1, dtype=np.int64)
    for e in range(E):
        for tile in range(starts[e] // block_m, (starts[e] + padded[e]) // block_m):
            expert_ids[tile] = e
    return sorted_ids, expert_ids, total, counts


# ----------------------------------------------------------------------------- experts

def silu(z):
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def expert_ffn(xrows, W13e, W2e) -> np.ndarray:
    """[P2 §1] one SwiGLU expert on a block of rows: W2 (silu(W1 x) * (W3 x)), with
    W1 = W13e[:I] (gate) and W3 = W13e[I:] (up) as in the §6 concatenation."""
    I = W2e.shape[1]
    h = f64(xrows) @ f64(W13e).T
    return (silu(h[:, :I]) * h[:, I:]) @ f64(W2e).T


def _expert(W, e):
    """Expert slice as float64; bf16 weights may be passed as uint16 bit arrays."""
    a = W[e]
    a = np.asarray(a)
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else f64(a)


def apply_expert_map(expert_ids, expert_map):
    """[P2 §10, "Try this": expert parallelism] relabel each tile of the align table with the
    local weight slot of its expert, or -1 when the expert is not on this device (its tiles
    are skipped)."""
    eid = np.asarray(expert_ids, dtype=np.int64).copy()
    m = np.asarray(expert_map, dtype=np.int64)
    valid = eid >= 0
    eid[valid] = m[eid[valid]]
    return eid


def moe_loop(x, ids, w, W13, W2, tokens=None, expert_map=None) -> np.ndarray:
    """Version A [P2 §3 moe_loop]: for each expert, gather the (token, slot) pairs routed
    to it in ascending flat row, run the expert once on those token rows, and add the
    weighted outputs back at their tokens. Experts with no rows are skipped.

    ``tokens`` restricts the computation to a subset of tokens (rows of the result
    follow that subset's order); the result for a token depends only on that token.
    ``expert_map`` (expert parallelism): expert e uses weight slot expert_map[e], and an
    expert mapped to -1 lives on another device and contributes nothing here.
    """
    x = f64(x)
    ids = np.asarray(ids, dtype=np.int64)
    w = f64(w)
    if tokens is None:
        tokens = np.arange(x.shape[0])
    tokens = np.asarray(tokens, dtype=np.int64)
    sub_ids, sub_w = ids[tokens], w[tokens]
    H = x.shape[1]
    out = np.zeros((tokens.size, H))
    E = int(max(W13.shape[0], sub_ids.max() + 1 if sub_ids.size else 0))
    for e in range(E):
        t_local, slot = np.nonzero(sub_ids == e)
        if t_local.size == 0:
            continue
        we = e if expert_map is None else int(expert_map[e])
        if we < 0:
            continue
        ye = expert_ffn(x[tokens[t_local]], _expert(W13, we), _expert(W2, we))
        np.add.at(out, t_local, ye * sub_w[t_local, slot][:, None])
    return out


def masked_forward(x_masked, counts, W13, W2, row_w=None) -> np.ndarray:
    """[P2 §9, DeepGEMM's "masked" layout; §7 fixed-capacity layouts for CUDA-graph decode]
    tokens already bucketed per expert: x_masked[E, C, H] with counts[e] valid rows in
    expert e's bucket. y[e, i] = row_w[e, i] * expert_e(x[e, i]) for i < counts[e]; rows past
    the count are not computed (returned as NaN here, "not written")."""
    x = f64(x_masked)
    E, C, H = x.shape
    y = np.full((E, C, H), np.nan)
    for e in range(E):
        n = int(counts[e])
        if n == 0:
            continue
        ye = expert_ffn(x[e, :n], _expert(W13, e), _expert(W2, e))
        wv = np.ones(n) if row_w is None else f64(row_w)[e, :n]
        y[e, :n] = ye * wv[:, None]
    return y


def dispatch_masked(x, ids, w, E, capacity):
    """Bucket the routed (token, slot) rows by expert, in ascending flat row, into a
    fixed-capacity layout (the expert-parallel dispatch a masked layout stands for).
    Returns x_masked[E, C, H], row_w[E, C], counts[E] and the (t, j) of every bucket row."""
    x = f64(x)
    T, k = ids.shape
    xm = np.zeros((E, capacity, x.shape[1]))
    wm = np.zeros((E, capacity))
    counts = np.zeros(E, dtype=np.int64)
    where = np.full((E, capacity, 2), -1, dtype=np.int64)
    for r in range(T * k):
        t, j = divmod(r, k)
        e = int(ids[t, j])
        i = counts[e]
        if i >= capacity:
            raise ValueError("capacity exceeded")
        xm[e, i], wm[e, i], where[e, i] = x[t], w[t, j], (t, j)
        counts[e] += 1
    return xm, wm, counts, where


def moe_dense(x, ids, w, W13, W2) -> np.ndarray:
    """Version B [P2 §3 moe_dense]: run EVERY expert on EVERY token, then combine with a
    [T, E] gate matrix holding the k routed weights per token (zeros elsewhere).
    E/k times the FLOPs of version A; shares no indexing code with it."""
    x = f64(x)
    T = x.shape[0]
    E = W13.shape[0]
    gate = np.zeros((T, E))
    for t in range(T):
        for j in range(ids.shape[1]):
            gate[t, int(ids[t, j])] += float(w[t, j])
    out = np.zeros_like(x)
    for e in range(E):
        out += gate[:, e:e + 1] * expert_ffn(x, _expert(W13, e), _expert(W2, e))
    return out


def add_shared_experts(ids, w, E, n_shared):
    """[P2 §1 model table: DeepSeek-V3 and Kimi K2 have 256 / 384 routed experts "+1
    shared"] a shared expert runs on every token with weight 1, outside the router: append
    slots k..k+n_shared-1 holding experts E..E+n_shared-1 (their weights follow the routed
    experts' in W13/W2)."""
    T = ids.shape[0]
    sid = np.broadcast_to(np.arange(E, E + n_shared), (T, n_shared))
    return (np.concatenate([ids, sid], axis=1),
            np.concatenate([w, np.ones((T, n_shared))], axis=1))


def moe_forward(x, Wg, W13, W2, k, mode=SOFTMAX, renormalize=True, scale=1.0,
                n_group=1, topk_group=1, logit_bias=None, select_bias=None, dense=False,
                n_shared=0):
    """Route then run version A (or B). Returns (out, ids, w, logits); with shared experts,
    ids/w include their slots."""
    logits = router_logits(x, Wg, logit_bias if mode == SOFTMAX else None)
    ids, w = route(logits, k, mode, renormalize, scale, n_group, topk_group, select_bias)
    if n_shared:
        ids, w = add_shared_experts(ids, w, Wg.shape[0], n_shared)
    out = (moe_dense if dense else moe_loop)(x, ids, w, W13, W2)
    return out, ids, w, logits


# ----------------------------------------------------------------------------- brute force

def brute_topk(keys_row, k):
    """Best k-subset by enumeration: maximise the sorted key vector lexicographically,
    preferring lower ids on exact ties. Returns ids in descending key order."""
    n = len(keys_row)
    best = None
    for comb in itertools.combinations(range(n), k):
        key = sorted(((keys_row[i], -i) for i in comb), reverse=True)
        if best is None or key > best[0]:
            best = (key, comb)
    return np.array([-i for _, i in best[0]], dtype=np.int64)


def brute_align(topk_ids, block_m, E):
    """sorted_ids / expert_ids / total by an independent route: sort (expert, r) pairs,
    then walk the experts and append each run followed by its sentinel padding."""
    flat = [int(e) for e in np.asarray(topk_ids).reshape(-1)]
    n = len(flat)
    pairs = sorted((e, r) for r, e in enumerate(flat))
    sorted_ids, expert_ids = [], []
    for e in range(E):
        run = [r for (ee, r) in pairs if ee == e]
        if not run:
            continue
        pad = (-len(run)) % block_m
        run = run + [n] * pad
        sorted_ids += run
        expert_ids += [e] * (len(run) // block_m)
    return np.array(sorted_ids, dtype=np.int64), np.array(expert_ids, dtype=np.int64), len(sorted_ids)
