"""Seeded synthetic workloads of the MoE expert layer.

This module only draws random numbers and holds the five workload shapes; it
contains none of the layer's arithmetic, so both the CUDA path and the CPU
oracle may take their inputs from it.

Recipe (per workload, ``seed`` fixed below):
  * one ``torch.Generator('cpu')`` seeded with ``seed`` draws, in order,
    x = randn[T, H] (float32, cast to BF16 with nearest-even) and then
    logits = randn[T, E] (float32);
  * the skewed prefill adds log(p_e) to column e of the logits, with
    p_e proportional to (e + 1) ** -1.2 (a Zipf popularity, expert 0 hottest);
  * expert e's weights come from their own generator seeded with
    ``expert_seed(seed, e)`` on the device asked for: l1_w[e] = randn[2I, H] * sigma,
    then l2_w[e] = randn[H, I] * sigma, both cast to BF16.  Per-expert
    generators let any single expert be regenerated without drawing the rest.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int        # tokens
    H: int        # hidden
    I: int        # intermediate (gate and up have I rows each)
    E: int        # experts
    k: int        # top-k
    sigma: float  # weight standard deviation
    seed: int
    zipf_s: float = 0.0   # > 0: add log(Zipf(s) popularity) to the logits

    @property
    def pairs(self) -> int:
        return self.T * self.k

    def describe(self) -> str:
        return (f"{self.name} T={self.T} H={self.H} I={self.I} E={self.E} k={self.k}")


WORKLOADS = {
    "tiny": Workload("tiny", T=64, H=256, I=128, E=8, k=2, sigma=0.02, seed=0),
    "small_decode": Workload("small_decode", T=8, H=2048, I=512, E=256, k=8, sigma=0.02, seed=1),
    "large_decode": Workload("large_decode", T=128, H=7168, I=2048, E=256, k=8, sigma=0.01, seed=2),
    "prefill": Workload("prefill", T=4096, H=7168, I=2048, E=256, k=8, sigma=0.01, seed=3),
    "skewed_prefill": Workload("skewed_prefill", T=8192, H=7168, I=2048, E=256, k=8, sigma=0.01,
                               seed=4, zipf_s=1.2),
}

# Smaller cases with the same per-expert shapes, for profiler captures that
# must stay small: the prefill's ~128 pairs per expert on 32 experts, the
# skewed prefill's popularity on 64 experts (hot experts of ~2000 pairs, i.e.
# ten 208-token tiles, a few experts with fewer than ten pairs; 1.5 GB of
# weights instead of 6).
PROFILE_WORKLOADS = {
    "prefill_e32": Workload("prefill_e32", T=512, H=7168, I=2048, E=32, k=8, sigma=0.01, seed=3),
    "skewed_e64": Workload("skewed_e64", T=2048, H=7168, I=2048, E=64, k=8, sigma=0.01, seed=4, zipf_s=1.2),
    # the large decode's ~4 pairs per expert on 32 experts (0.75 GB of weights)
    "large_decode_e32": Workload("large_decode_e32", T=16, H=7168, I=2048, E=32, k=8, sigma=0.01, seed=2),
}


def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """Bit patterns (int16 view) of a BF16 tensor."""
    assert t.dtype == torch.bfloat16
    return t.view(torch.int16)


def tokens(wl: Workload):
    """(x bf16 [T, H], logits float32 [T, E]) on the CPU."""
    g = torch.Generator(device="cpu").manual_seed(wl.seed)
    x = torch.randn(wl.T, wl.H, generator=g, dtype=torch.float32).to(torch.bfloat16)
    logits = torch.randn(wl.T, wl.E, generator=g, dtype=torch.float32)
    if wl.zipf_s > 0:
        ranks = np.arange(1, wl.E + 1, dtype=np.float64)
        p = ranks ** -wl.zipf_s
        p /= p.sum()
        logits = logits + torch.from_numpy(np.log(p)).to(torch.float32)[None, :]
    return x, logits


def expert_seed(seed: int, e: int) -> int:
    return (seed + 1) * 1_000_003 + e


def expert_weights(wl: Workload, e: int, device="cpu"):
    """(l1_w bf16 [2I, H], l2_w bf16 [H, I]) of expert e, drawn on ``device``."""
    g = torch.Generator(device=device).manual_seed(expert_seed(wl.seed, e))
    l1 = torch.randn(2 * wl.I, wl.H, generator=g, device=device, dtype=torch.float32)
    l1 = (l1 * wl.sigma).to(torch.bfloat16)
    l2 = torch.randn(wl.H, wl.I, generator=g, device=device, dtype=torch.float32)
    l2 = (l2 * wl.sigma).to(torch.bfloat16)
    return l1, l2


def all_expert_weights(wl: Workload, device="cpu"):
    """Stacked (l1_w [E, 2I, H], l2_w [E, H, I]) BF16 -- only for small workloads."""
    l1s, l2s = zip(*(expert_weights(wl, e, device) for e in range(wl.E)))
    return torch.stack(l1s), torch.stack(l2s)


def zipf_popularity(E: int, s: float) -> np.ndarray:
    p = np.arange(1, E + 1, dtype=np.float64) ** -s
    return p / p.sum()


def bytes_of(wl: Workload) -> dict:
    """Sizes used by the roofline: weights per expert (FP4 + UE8M0) and activations."""
    w_elems = 3 * wl.H * wl.I
    return {
        "weight_bytes_per_expert": w_elems // 2 + w_elems // 32,
        "x_bytes": wl.T * wl.H * 2,
        "logits_bytes": wl.T * wl.E * 4,
        "y_bytes": wl.T * wl.H * 2,
        "flops": 2 * wl.pairs * 3 * wl.H * wl.I,
    }


__all__ = ["Workload", "WORKLOADS", "tokens", "expert_weights", "all_expert_weights",
           "bf16_bits", "expert_seed", "bytes_of", "zipf_popularity", "math"]
