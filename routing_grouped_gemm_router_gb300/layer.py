"""MoELayer: owns the workspace of one layer shape and calls the C ABI's moe_forward.

PyTorch provides the device memory (caching allocator) and the stream; the layer itself
runs in libmoe_gb300.so.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib as L


class MoELayer:
    """A fused MoE feed-forward layer with caller-provided weights.

    x[T,H], Wg[E,H], W13[E,2I,H] (gate rows 0..I-1, up rows I..2I-1), W2[E,H,I] in one
    dtype (bf16 or fp32), all on one CUDA device. ``forward`` enqueues the whole layer on
    the current stream without a host round-trip.

    FP8 expert weights: W13/W2 hold E4M3 codes (torch.float8_e4m3fn or uint8) and
    w13_scale[E', 2, ceil(I/128), ceil(H/128)], w2_scale[E', ceil(H/128), ceil(I/128)] the
    fp32 scale of each 128 x 128 block (E' = E + n_shared); x and Wg stay bf16.
    """

    def __init__(self, Wg, W13, W2, k, mode=L.MOE_ROUTE_SOFTMAX, renormalize=True, scale=1.0,
                 n_group=1, topk_group=1, logit_bias: Optional[torch.Tensor] = None,
                 select_bias: Optional[torch.Tensor] = None,
                 expert_map: Optional[torch.Tensor] = None, n_shared: int = 0,
                 w13_scale: Optional[torch.Tensor] = None,
                 w2_scale: Optional[torch.Tensor] = None):
        """W13/W2 hold E routed experts followed by n_shared shared experts."""
        if (w13_scale is None) != (w2_scale is None):
            raise ValueError("FP8 weights need both w13_scale and w2_scale")
        self.w13_scale = w13_scale.float().contiguous() if w13_scale is not None else None
        self.w2_scale = w2_scale.float().contiguous() if w2_scale is not None else None
        self.Wg, self.W13, self.W2 = Wg, W13, W2
        self.E, self.H = Wg.shape
        self.n_shared = n_shared
        self.I = W2.shape[2]
        self.k = k
        self.dtype = {torch.bfloat16: L.MOE_BF16, torch.float32: L.MOE_F32}[Wg.dtype]
        self.mode, self.renormalize, self.scale = mode, renormalize, scale
        self.n_group, self.topk_group = n_group, topk_group
        self.logit_bias = logit_bias.float().contiguous() if logit_bias is not None else None
        self.select_bias = select_bias.float().contiguous() if select_bias is not None else None
        self.expert_map = (expert_map.to(torch.int32).contiguous()
                           if expert_map is not None else None)
        self._ws = None
        self._ws_T = None

    def config(self, T):
        return L.make_config(T, self.H, self.I, self.E, self.k, self.dtype, self.mode,
                             self.renormalize, self.scale, self.n_group, self.topk_group,
                             self.logit_bias, self.select_bias, self.expert_map,
                             self.n_shared, self.w13_scale, self.w2_scale)

    def workspace(self, T):
        if self._ws_T != T:
            cfg = self.config(T)
            self._layout = L.moe_workspace_layout(cfg)
            self._ws = torch.empty(self._layout.total, dtype=torch.uint8, device=self.Wg.device)
            self._ws_T = T
        return self._ws, self._layout

    def forward(self, x, out=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        ws, layout = self.workspace(T)
        L.moe_forward(self.config(T), x, self.Wg, self.W13, self.W2, out, ws, layout.total)
        return out

    __call__ = forward

    # Views of the intermediates the last forward left in the workspace (tests, debugging).
    def intermediates(self, T):
        ws, lay = self.workspace(T)
        kk = self.k + self.n_shared
        n = T * kk
        dt = self.Wg.dtype

        def view(off, count, dtype):
            esz = torch.tensor([], dtype=dtype).element_size()
            return ws[off:off + count * esz].view(dtype)

        return {
            "logits": view(lay.logits, T * self.E, torch.float32).view(T, self.E),
            "topk_ids": view(lay.topk_ids, n, torch.int32).view(T, kk),
            "topk_w": view(lay.topk_w, n, torch.float32).view(T, kk),
            "sorted_ids": view(lay.sorted_ids, lay.max_padded, torch.int32),
            "expert_ids": view(lay.expert_ids, lay.max_padded // lay.block_m, torch.int32),
            "num_post_padded": view(lay.num_post_padded, 1, torch.int32),
            "counts": view(lay.counts, self.E + self.n_shared, torch.int32),
            "y": view(lay.y, n * self.H, dt).view(n, self.H),
            "block_m": lay.block_m,
            "max_padded": lay.max_padded,
        }
