"""ctypes binding of libmoe_gb300.so: the C ABI of include/moe.h under the same names.

Argument marshalling only: tensors become device pointers (``data_ptr()``), streams become
``cudaStream_t`` handles, and a non-OK status raises ``MoeError``. Every step of the layer
runs in the library's CUDA kernels; there is no Python or CPU fallback, and importing this
module fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA = range(5)
MOE_F32, MOE_BF16 = 0, 1
MOE_ROUTE_SOFTMAX, MOE_ROUTE_SIGMOID_GROUPED = 0, 1
MOE_WEIGHTS_NATIVE, MOE_WEIGHTS_FP8_E4M3_B128 = 0, 1


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


class moe_config_t(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("E", ctypes.c_int), ("k", ctypes.c_int), ("dtype", ctypes.c_int),
                ("mode", ctypes.c_int), ("renormalize", ctypes.c_int), ("scale", ctypes.c_float),
                ("n_group", ctypes.c_int), ("topk_group", ctypes.c_int),
                ("logit_bias", ctypes.c_void_p), ("select_bias", ctypes.c_void_p),
                ("expert_map", ctypes.c_void_p), ("n_shared", ctypes.c_int),
                ("weight_format", ctypes.c_int), ("w13_scale", ctypes.c_void_p),
                ("w2_scale", ctypes.c_void_p)]


class moe_ws_layout_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("logits", "topk_ids", "topk_w", "sorted_ids",
                                              "expert_ids", "num_post_padded", "counts",
                                              "align_scratch", "act", "xs", "y", "gemm_scratch",
                                              "total")] + \
               [("block_m", ctypes.c_int), ("max_padded", ctypes.c_int)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m routing_grouped_gemm_router_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, SZ, ST = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_int
    CFG = ctypes.POINTER(moe_config_t)
    sig = {
        "moe_abi_version": (I32, []),
        "moe_status_string": (ctypes.c_char_p, [ST]),
        "moe_block_m": (I32, [CFG]),
        "moe_small_batch": (I32, [CFG]),
        "moe_gemm_kernel": (I32, [CFG]),
        "moe_max_padded_rows": (SZ, [I32, I32, I32, I32]),
        "moe_align_workspace_size": (ST, [I32, I32, I32, I32, ctypes.POINTER(SZ)]),
        "moe_workspace_layout": (ST, [CFG, ctypes.POINTER(moe_ws_layout_t)]),
        "moe_workspace_size": (ST, [CFG, ctypes.POINTER(SZ)]),
        "moe_route": (ST, [CFG, P, P, P, P, P, P]),
        "moe_align": (ST, [P, I32, I32, I32, I32, P, P, P, P, P, SZ, P]),
        "moe_align_noalloc": (ST, [P, I32, I32, I32, I32, P, P, P, P, P]),
        "moe_expert_gemm1_workspace_size": (ST, [CFG, I32, ctypes.POINTER(SZ)]),
        "moe_expert_gemm1": (ST, [CFG, P, P, P, P, P, I32, P, P, SZ, P]),
        "moe_gather_rows": (ST, [P, P, P, I32, I32, I32, I32, P, P]),
        "moe_expert_gemm1_gathered_workspace_size": (ST, [CFG, I32, ctypes.POINTER(SZ)]),
        "moe_expert_gemm1_gathered": (ST, [CFG, P, P, P, P, P, I32, P, P, SZ, P]),
        "moe_expert_gemm2_workspace_size": (ST, [CFG, I32, ctypes.POINTER(SZ)]),
        "moe_grouped_swiglu_workspace_size": (ST, [CFG, I32, ctypes.POINTER(SZ)]),
        "moe_expert_gemm2": (ST, [CFG, P, P, P, P, P, I32, P, P, P, SZ, P]),
        "moe_grouped_swiglu": (ST, [CFG, P, P, P, P, P, P, I32, P, P, P, SZ, P]),
        "moe_combine": (ST, [P, I32, I32, I32, I32, P, P]),
        "moe_apply_expert_map": (ST, [P, I32, P, I32, P]),
        "moe_masked_table": (ST, [P, I32, I32, I32, P, P, P, P]),
        "moe_masked_workspace_size": (ST, [CFG, I32, ctypes.POINTER(SZ)]),
        "moe_masked_forward": (ST, [CFG, P, P, I32, P, P, P, P, P, SZ, P]),
        "moe_combine_local": (ST, [P, P, P, I32, I32, I32, I32, I32, P, P]),
        "moe_forward": (ST, [CFG, P, P, P, P, P, P, SZ, P]),
        "moe_device_status": (I32, [I32]),
        "moe_selftest_wait_timeout": (ST, [P]),
        "moe_route_logits": (ST, [CFG, P, P, P, P]),
        "moe_dequant_fp8_weights": (ST, [CFG, I32, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


_lib = _load()
EXPORTED = ("moe_abi_version", "moe_status_string", "moe_block_m", "moe_small_batch",
            "moe_gemm_kernel",
            "moe_max_padded_rows",
            "moe_align_workspace_size", "moe_workspace_layout", "moe_workspace_size",
            "moe_route", "moe_align", "moe_align_noalloc", "moe_expert_gemm1_workspace_size",
            "moe_expert_gemm1", "moe_gather_rows", "moe_expert_gemm1_gathered_workspace_size",
            "moe_expert_gemm1_gathered", "moe_grouped_swiglu_workspace_size",
            "moe_expert_gemm2_workspace_size", "moe_expert_gemm2",
            "moe_grouped_swiglu", "moe_combine", "moe_apply_expert_map", "moe_combine_local",
            "moe_masked_table", "moe_masked_workspace_size", "moe_masked_forward",
            "moe_forward", "moe_device_status", "moe_selftest_wait_timeout",
            "moe_route_logits", "moe_dequant_fp8_weights")


def lib():
    return _lib


# ---------------------------------------------------------------------------- marshalling

def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn, st):
    if st != MOE_OK:
        raise MoeError(fn, st)


def status_string(st: int) -> str:
    return _lib.moe_status_string(st).decode()


def make_config(T, H, I, E, k, dtype=MOE_BF16, mode=MOE_ROUTE_SOFTMAX, renormalize=True,
                scale=1.0, n_group=1, topk_group=1, logit_bias=None, select_bias=None,
                expert_map=None, n_shared=0, w13_scale=None, w2_scale=None):
    """Build a ``moe_config_t``; biases (fp32), expert_map (int32) and the FP8 block scales
    (fp32) are device tensors the caller keeps alive. Passing both scales selects FP8
    E4M3 expert weights (W13/W2 then hold the codes as uint8 / float8_e4m3fn)."""
    fp8 = w13_scale is not None or w2_scale is not None
    return moe_config_t(T, H, I, E, k, dtype, mode, int(bool(renormalize)), float(scale),
                        n_group, topk_group, _ptr(logit_bias), _ptr(select_bias),
                        _ptr(expert_map), int(n_shared),
                        MOE_WEIGHTS_FP8_E4M3_B128 if fp8 else MOE_WEIGHTS_NATIVE,
                        _ptr(w13_scale), _ptr(w2_scale))


def moe_selftest_wait_timeout(stream=None):
    """Diagnostic: a CTA whose pipeline waits time out (see include/moe.h); afterwards
    moe_device_status() reads 2."""
    _check("moe_selftest_wait_timeout", _lib.moe_selftest_wait_timeout(_stream(stream)))


def moe_abi_version() -> int:
    return _lib.moe_abi_version()


def moe_block_m(cfg) -> int:
    return _lib.moe_block_m(ctypes.byref(cfg))


def moe_small_batch(cfg) -> bool:
    """Whether the grouped GEMMs of cfg run as the small-batch (decode) kernels."""
    return bool(_lib.moe_small_batch(ctypes.byref(cfg)))


MOE_GEMM_INVALID, MOE_GEMM_SIMT, MOE_GEMM_SMALL_BATCH, MOE_GEMM_DECODE_TC, MOE_GEMM_PAIR_TC = range(5)


def moe_gemm_kernel(cfg) -> int:
    """Which kernels run the grouped GEMMs of cfg (one of the MOE_GEMM_* values)."""
    return _lib.moe_gemm_kernel(ctypes.byref(cfg))


def moe_max_padded_rows(T, k, E, block_m) -> int:
    return _lib.moe_max_padded_rows(T, k, E, block_m)


def moe_align_workspace_size(T, k, E, block_m) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_align_workspace_size", _lib.moe_align_workspace_size(T, k, E, block_m, ctypes.byref(out)))
    return out.value


def moe_workspace_layout(cfg) -> moe_ws_layout_t:
    out = moe_ws_layout_t()
    _check("moe_workspace_layout", _lib.moe_workspace_layout(ctypes.byref(cfg), ctypes.byref(out)))
    return out


def moe_workspace_size(cfg) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_workspace_size", _lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(out)))
    return out.value


def moe_route_logits(cfg, x, Wg, logits, stream=None):
    _check("moe_route_logits", _lib.moe_route_logits(ctypes.byref(cfg), _ptr(x), _ptr(Wg),
                                                     _ptr(logits), _stream(stream)))


def moe_route(cfg, x, Wg, logits, topk_ids, topk_w, stream=None):
    _check("moe_route", _lib.moe_route(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(logits),
                                       _ptr(topk_ids), _ptr(topk_w), _stream(stream)))


def moe_align(topk_ids, T, k, E, block_m, sorted_ids, expert_ids, num_post_padded,
              counts=None, ws=None, ws_bytes=0, stream=None):
    _check("moe_align", _lib.moe_align(_ptr(topk_ids), T, k, E, block_m, _ptr(sorted_ids),
                                       _ptr(expert_ids), _ptr(num_post_padded), _ptr(counts),
                                       _ptr(ws), ws_bytes, _stream(stream)))


def moe_align_noalloc(topk_ids, T, k, E, block_m, sorted_ids, expert_ids, num_post_padded,
                      counts=None, stream=None):
    """moe_align for callers that cannot provide scratch memory (see include/moe.h)."""
    _check("moe_align_noalloc", _lib.moe_align_noalloc(
        _ptr(topk_ids), T, k, E, block_m, _ptr(sorted_ids), _ptr(expert_ids),
        _ptr(num_post_padded), _ptr(counts), _stream(stream)))


def moe_expert_gemm1_workspace_size(cfg, block_m) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_expert_gemm1_workspace_size",
           _lib.moe_expert_gemm1_workspace_size(ctypes.byref(cfg), block_m, ctypes.byref(out)))
    return out.value


def moe_expert_gemm1_gathered_workspace_size(cfg, block_m) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_expert_gemm1_gathered_workspace_size",
           _lib.moe_expert_gemm1_gathered_workspace_size(ctypes.byref(cfg), block_m,
                                                         ctypes.byref(out)))
    return out.value


def moe_expert_gemm2_workspace_size(cfg, block_m) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_expert_gemm2_workspace_size",
           _lib.moe_expert_gemm2_workspace_size(ctypes.byref(cfg), block_m, ctypes.byref(out)))
    return out.value


def moe_grouped_swiglu_workspace_size(cfg, block_m) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_grouped_swiglu_workspace_size",
           _lib.moe_grouped_swiglu_workspace_size(ctypes.byref(cfg), block_m, ctypes.byref(out)))
    return out.value


def moe_expert_gemm1(cfg, x, W13, sorted_ids, expert_ids, num_post_padded, block_m, act,
                     ws=None, ws_bytes=0, stream=None):
    _check("moe_expert_gemm1", _lib.moe_expert_gemm1(
        ctypes.byref(cfg), _ptr(x), _ptr(W13), _ptr(sorted_ids), _ptr(expert_ids),
        _ptr(num_post_padded), block_m, _ptr(act), _ptr(ws), ws_bytes, _stream(stream)))


def moe_dequant_fp8_weights(cfg, matrix, codes, counts, out, stream=None):
    """FP8 codes of W13 (matrix 1) or W2 (matrix 2) times their block scales as bf16 weights."""
    _check("moe_dequant_fp8_weights", _lib.moe_dequant_fp8_weights(
        ctypes.byref(cfg), matrix, _ptr(codes), _ptr(counts), _ptr(out), _stream(stream)))


def moe_gather_rows(x, sorted_ids, num_post_padded, T, k, H, dtype, xs, stream=None):
    _check("moe_gather_rows", _lib.moe_gather_rows(
        _ptr(x), _ptr(sorted_ids), _ptr(num_post_padded), T, k, H, dtype, _ptr(xs),
        _stream(stream)))


def moe_expert_gemm1_gathered(cfg, xs, W13, sorted_ids, expert_ids, num_post_padded, block_m,
                              act, ws=None, ws_bytes=0, stream=None):
    _check("moe_expert_gemm1_gathered", _lib.moe_expert_gemm1_gathered(
        ctypes.byref(cfg), _ptr(xs), _ptr(W13), _ptr(sorted_ids), _ptr(expert_ids),
        _ptr(num_post_padded), block_m, _ptr(act), _ptr(ws), ws_bytes, _stream(stream)))


def moe_expert_gemm2(cfg, act, W2, sorted_ids, expert_ids, num_post_padded, block_m, topk_w, y,
                     ws=None, ws_bytes=0, stream=None):
    _check("moe_expert_gemm2", _lib.moe_expert_gemm2(
        ctypes.byref(cfg), _ptr(act), _ptr(W2), _ptr(sorted_ids), _ptr(expert_ids),
        _ptr(num_post_padded), block_m, _ptr(topk_w), _ptr(y), _ptr(ws), ws_bytes,
        _stream(stream)))


def moe_grouped_swiglu(cfg, x, W13, W2, sorted_ids, expert_ids, num_post_padded, block_m,
                       topk_w, y, ws, ws_bytes, stream=None):
    _check("moe_grouped_swiglu", _lib.moe_grouped_swiglu(
        ctypes.byref(cfg), _ptr(x), _ptr(W13), _ptr(W2), _ptr(sorted_ids), _ptr(expert_ids),
        _ptr(num_post_padded), block_m, _ptr(topk_w), _ptr(y), _ptr(ws), ws_bytes,
        _stream(stream)))


def moe_combine(y, T, k, H, dtype, out, stream=None):
    _check("moe_combine", _lib.moe_combine(_ptr(y), T, k, H, dtype, _ptr(out), _stream(stream)))


def moe_apply_expert_map(expert_ids, num_tiles, expert_map, E, stream=None):
    _check("moe_apply_expert_map", _lib.moe_apply_expert_map(
        _ptr(expert_ids), num_tiles, _ptr(expert_map), E, _stream(stream)))


def moe_combine_local(y, topk_ids, expert_map, E, T, k, H, dtype, out, stream=None):
    _check("moe_combine_local", _lib.moe_combine_local(
        _ptr(y), _ptr(topk_ids), _ptr(expert_map), E, T, k, H, dtype, _ptr(out),
        _stream(stream)))


def moe_masked_table(counts, E, capacity, block_m, sorted_ids, expert_ids, num_post_padded,
                     stream=None):
    _check("moe_masked_table", _lib.moe_masked_table(
        _ptr(counts), E, capacity, block_m, _ptr(sorted_ids), _ptr(expert_ids),
        _ptr(num_post_padded), _stream(stream)))


def moe_masked_workspace_size(cfg, capacity) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_masked_workspace_size",
           _lib.moe_masked_workspace_size(ctypes.byref(cfg), capacity, ctypes.byref(out)))
    return out.value


def moe_masked_forward(cfg, x_masked, counts, capacity, row_w, W13, W2, y_masked, ws, ws_bytes,
                       stream=None):
    _check("moe_masked_forward", _lib.moe_masked_forward(
        ctypes.byref(cfg), _ptr(x_masked), _ptr(counts), capacity, _ptr(row_w), _ptr(W13),
        _ptr(W2), _ptr(y_masked), _ptr(ws), ws_bytes, _stream(stream)))


def moe_forward(cfg, x, Wg, W13, W2, out, ws, ws_bytes, stream=None):
    _check("moe_forward", _lib.moe_forward(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(W13),
                                           _ptr(W2), _ptr(out), _ptr(ws), ws_bytes,
                                           _stream(stream)))


def moe_device_status(reset=True) -> int:
    return _lib.moe_device_status(int(bool(reset)))
