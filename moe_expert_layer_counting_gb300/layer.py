"""Device-side containers around the C ABI: quantised expert weights and a
layer object that owns its workspace.  Allocation uses torch; every
computation is a call into libmoe_mxq.so."""
from __future__ import annotations

import torch

from . import binding as B


class QuantizedExperts:
    """FP4 E2M1 + UE8M0 expert weights in the MMA layouts the GEMMs read.

    w1q [E, 2I, H/2] / w1s (E*2I*H/32 bytes, chunk order) -- gate/up interleaved by 8;
    w2q [E, H, I/2]  / w2s (E*H*I/32 bytes, chunk order).
    """

    def __init__(self, E: int, H: int, I: int, device="cuda"):
        self.E, self.H, self.I = E, H, I
        self.w1q = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=device)
        self.w1s = torch.empty(E * 2 * I * H // 32, dtype=torch.uint8, device=device)
        self.w2q = torch.empty(E, H, I // 2, dtype=torch.uint8, device=device)
        self.w2s = torch.empty(E * H * I // 32, dtype=torch.uint8, device=device)

    def set_expert(self, e: int, l1_w: torch.Tensor, l2_w: torch.Tensor, stream=None):
        """Quantise expert e from BF16 l1_w [2I, H] (gate rows then up rows) and l2_w [H, I]."""
        H, I = self.H, self.I
        assert l1_w.shape == (2 * I, H) and l2_w.shape == (H, I)
        s1 = 2 * I * H // 32
        s2 = H * I // 32
        B.mxq_quantize_weight(l1_w.contiguous().view(1, 2 * I, H), B.LAYOUT_MMA_L1, self.w1q[e],
                              self.w1s[e * s1:(e + 1) * s1], stream)
        B.mxq_quantize_weight(l2_w.contiguous().view(1, H, I), B.LAYOUT_MMA_L2, self.w2q[e],
                              self.w2s[e * s2:(e + 1) * s2], stream)

    @classmethod
    def from_bf16(cls, l1_w: torch.Tensor, l2_w: torch.Tensor, stream=None):
        E, twoI, H = l1_w.shape
        q = cls(E, H, twoI // 2, device=l1_w.device)
        B.mxq_quantize_weight(l1_w.contiguous(), B.LAYOUT_MMA_L1, q.w1q, q.w1s, stream)
        B.mxq_quantize_weight(l2_w.contiguous(), B.LAYOUT_MMA_L2, q.w2q, q.w2s, stream)
        return q


class MoELayer:
    """The MoE expert layer for a fixed (max_tokens, H, I, E, k): y = layer(x, logits)."""

    def __init__(self, weights: QuantizedExperts, k: int, max_tokens: int, tile_n: int = 0,
                 route_mode: int = B.ROUTE_SOFTMAX, schedule: int = B.SCHEDULE_DEFAULT):
        self.w = weights
        self.k = k
        self.max_tokens = max_tokens
        self.tile_n = tile_n
        self.route_mode = route_mode
        self.schedule = schedule
        nbytes = B.moe_workspace_size(max_tokens, weights.H, weights.I, weights.E, k)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=weights.w1q.device)

    def __call__(self, x: torch.Tensor, logits: torch.Tensor, y: torch.Tensor = None, stream=None, **outs):
        T = x.shape[0]
        assert T <= self.max_tokens
        if y is None:
            y = torch.empty_like(x)
        w = self.w
        ws = self.workspace
        need = B.moe_workspace_size(T, w.H, w.I, w.E, self.k)
        B.moe_forward(x, logits, w.w1q, w.w1s, w.w2q, w.w2s, self.k, y, ws[:need], tile_n=self.tile_n,
                      route_mode=self.route_mode, schedule=self.schedule, stream=stream, **outs)
        return y

    def device_status(self, stream=None) -> int:
        return B.moe_get_device_status(self.workspace, stream)


class Bfp8Experts:
    """Block-FP8 expert weights: E4M3 codes (tile-contiguous by default) with
    one float32 scale per 128 x 128 block.

    w1q (E*2I*H bytes) / w1s [E, 2I/128, H/128] -- gate rows [0, I), up rows [I, 2I);
    w2q (E*H*I bytes)  / w2s [E, H/128, I/128].
    """

    def __init__(self, E: int, H: int, I: int, device="cuda", layout: int = B.BFP8_LAYOUT_TILED):
        self.E, self.H, self.I, self.layout = E, H, I, layout
        self.w1q = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=device)
        self.w1s = torch.empty(E, 2 * I // 128, H // 128, dtype=torch.float32, device=device)
        self.w2q = torch.empty(E, H, I, dtype=torch.uint8, device=device)
        self.w2s = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device=device)

    def set_expert(self, e: int, l1_w: torch.Tensor, l2_w: torch.Tensor, stream=None):
        """Quantise expert e from BF16 l1_w [2I, H] (gate rows then up rows) and l2_w [H, I]."""
        H, I = self.H, self.I
        assert l1_w.shape == (2 * I, H) and l2_w.shape == (H, I)
        B.bfp8_quantize_weight(l1_w.contiguous().view(1, 2 * I, H), self.w1q[e:e + 1], self.w1s[e:e + 1],
                               self.layout, stream)
        B.bfp8_quantize_weight(l2_w.contiguous().view(1, H, I), self.w2q[e:e + 1], self.w2s[e:e + 1],
                               self.layout, stream)

    @classmethod
    def from_bf16(cls, l1_w: torch.Tensor, l2_w: torch.Tensor, layout: int = B.BFP8_LAYOUT_TILED, stream=None):
        E, twoI, H = l1_w.shape
        q = cls(E, H, twoI // 2, device=l1_w.device, layout=layout)
        B.bfp8_quantize_weight(l1_w.contiguous(), q.w1q, q.w1s, layout, stream)
        B.bfp8_quantize_weight(l2_w.contiguous(), q.w2q, q.w2s, layout, stream)
        return q


class MoELayerBfp8:
    """The block-FP8 MoE expert layer for a fixed (max_tokens, H, I, E, k): y = layer(x, logits)."""

    def __init__(self, weights: Bfp8Experts, k: int, max_tokens: int, route_mode: int = B.ROUTE_SOFTMAX):
        self.w = weights
        self.k = k
        self.max_tokens = max_tokens
        self.route_mode = route_mode
        nbytes = B.moe_bfp8_workspace_size(max_tokens, weights.H, weights.I, weights.E, k)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=weights.w1q.device)

    def __call__(self, x: torch.Tensor, logits: torch.Tensor, y: torch.Tensor = None, stream=None, **outs):
        T = x.shape[0]
        assert T <= self.max_tokens
        if y is None:
            y = torch.empty_like(x)
        w = self.w
        need = B.moe_bfp8_workspace_size(T, w.H, w.I, w.E, self.k)
        B.moe_forward_bfp8(x, logits, w.w1q, w.w1s, w.w2q, w.w2s, self.k, y, self.workspace[:need],
                           route_mode=self.route_mode, weight_layout=w.layout, stream=stream, **outs)
        return y

    def device_status(self, stream=None) -> int:
        return B.moe_get_device_status(self.workspace, stream)
