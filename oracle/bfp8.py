"""Block-FP8 variant of the MoE expert layer: plain CPU oracle (float64).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import or run this module.  It shares
no code with the CUDA library and never imports it.

The variant follows the single-kernel MoE of the MonoMoe kernel design page
("Fixed shape" and section 1, "Five-phase pipeline"): weights are E4M3 codes
with one scale per 128 x 128 block; the BF16 input is cast to FP8 with
per-token scales before the up-projection (phase 2); the up-projection is
followed by SiLU(gate) * up and a write-back to FP8 (phase 3); the
down-projection's FP32 partials of a token are summed (phase 4) and cast to
BF16 (phase 5).  Routing (softmax or sigmoid top-k, optional
renormalisation) and the counting-sort permute are the layer's own (``moe``).

Readings where the page leaves a step open:
  * every activation scale covers 128 consecutive values of one row along K
    (the x rows before GEMM1, the h rows before GEMM2), matching the weights'
    128-wide K blocks;
  * a scale is ``amax / 448`` computed in float32 (not rounded to a power of
    two); the codes are the E4M3 round-to-nearest-even of ``value / scale``
    computed in float32 -- the precision the kernels decide the codes in --
    clamped to +-448; a group whose amax is 0 has scale 0 and all codes 0;
  * the top-k weight multiplies each pair's float down-projection output, and
    the k weighted outputs of a token are summed, then rounded once to BF16
    (no per-pair BF16 rounding: the page accumulates FP32 partials).

Every floating-point step apart from those decisions is done in float64.
"""
from __future__ import annotations

import numpy as np

from . import formats as F
from . import moe

BLOCK = 128                       # K-block length of every scale, and weight rows per block
_F32_QMAX = np.float32(F.E4M3_MAX)


def _scale_and_codes(v32: np.ndarray, amax32: np.ndarray):
    """Scales ``amax / 448`` (float32) and E4M3 codes of ``v32 / scale`` (float32).

    ``v32`` [..., n] float32 values of groups whose float32 amax is ``amax32``
    [...]; zero groups get scale 0 and codes 0.
    """
    s = (amax32 / _F32_QMAX).astype(np.float32)
    nz = s > 0
    safe = np.where(nz, s, np.float32(1.0)).astype(np.float32)
    q = (v32 / safe[..., None]).astype(np.float32)             # float32 division, rounded once
    q = np.clip(q.astype(np.float64), -F.E4M3_MAX, F.E4M3_MAX)
    codes = np.where(nz[..., None], F.encode_e4m3(q), np.uint8(0)).astype(np.uint8)
    return s, codes


def quantize_rows(v: np.ndarray):
    """float64 [rows, K] -> (E4M3 codes uint8 [rows, K], float32 scales [rows, K/128]).

    One scale per 128 consecutive values of a row (the per-token activation
    scale of phases 2 and 3 of the MonoMoe kernel design).  The values are
    first rounded to float32 (exact for BF16 input).
    """
    rows, K = v.shape
    assert K % BLOCK == 0
    v32 = np.asarray(v, dtype=np.float64).astype(np.float32).reshape(rows, K // BLOCK, BLOCK)
    amax32 = np.max(np.abs(v32), axis=-1)
    s, codes = _scale_and_codes(v32, amax32)
    return codes.reshape(rows, K), s


def quantize_act(x_bf16_bits: np.ndarray):
    """BF16 [rows, K] -> (E4M3 codes [rows, K], float32 scales [rows, K/128])."""
    return quantize_rows(F.bf16_bits_to_f64(x_bf16_bits))


def quantize_weight(w_bf16_bits: np.ndarray):
    """BF16 [G, N, K] -> (E4M3 codes uint8 [G, N, K], float32 scales [G, N/128, K/128]).

    One scale per 128 x 128 block of each matrix (MonoMoe kernel design,
    "Fixed shape": block-FP8 (128 x 128) weights); codes in the natural
    row-major layout.
    """
    G, N, K = w_bf16_bits.shape
    assert N % BLOCK == 0 and K % BLOCK == 0
    w32 = F.bf16_bits_to_f64(w_bf16_bits).astype(np.float32)
    blocks = w32.reshape(G, N // BLOCK, BLOCK, K // BLOCK, BLOCK).transpose(0, 1, 3, 2, 4)
    blocks = blocks.reshape(G, N // BLOCK, K // BLOCK, BLOCK * BLOCK)
    amax32 = np.max(np.abs(blocks), axis=-1)
    s, codes = _scale_and_codes(blocks, amax32)
    codes = codes.reshape(G, N // BLOCK, K // BLOCK, BLOCK, BLOCK).transpose(0, 1, 3, 2, 4)
    return codes.reshape(G, N, K), s


def dequant_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """E4M3 codes [..., K] with float32 scales [..., K/128] -> float64."""
    v = F.decode_e4m3(codes)
    return v * np.repeat(scales.astype(np.float64), BLOCK, axis=-1)


def dequant_weight(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """E4M3 codes [N, K] with float32 block scales [N/128, K/128] -> float64 [N, K]."""
    s = np.repeat(np.repeat(scales.astype(np.float64), BLOCK, axis=0), BLOCK, axis=1)
    return F.decode_e4m3(codes) * s


# ---------------------------------------------------------------- expert GEMMs

def expert_forward(xq, xs, w1q, w1s, w2q, w2s, topk_idx, E: int, experts=None, return_h: bool = False):
    """Up-projection + SiLU(gate) * up + FP8 write-back + down-projection per pair.

    Weights in the natural layout: l1 [E, 2I, H] with gate rows [0, I) and up
    rows [I, 2I), l2 [E, H, I], each with 128 x 128 block scales.  For a pair
    p = (t, j) routed to expert e:

        acc    = deq(xq[t]) . deq(W1[e])^T            (2I values)
        h      = silu(acc[:I]) * acc[I:]              (I values, no weight)
        hq, hs = quantize_rows(h)                     (per 128 along I)
        y_p    = deq(hq, hs) . deq(W2[e])^T           (H values, kept in float64)

    Returns y_pairs float64 [k, T, H] (dropped pairs' rows 0) and, with
    ``return_h``, hq [P, I] / hs [P, I/128] indexed by pair id.
    """
    T, k = topk_idx.shape
    H = xq.shape[1]
    I = w2q.shape[2]
    y_pairs = np.zeros((k, T, H), dtype=np.float64)
    hq_all = np.zeros((T * k, I), dtype=np.uint8)
    hs_all = np.zeros((T * k, I // BLOCK), dtype=np.float32)
    flat = topk_idx.reshape(-1)
    todo = range(E) if experts is None else experts
    for e in todo:
        pairs = np.nonzero(flat == e)[0]
        if pairs.size == 0:
            continue
        tok = pairs // k
        slot = pairs % k
        X = dequant_rows(xq[tok], xs[tok])                        # [n, H]
        W1 = dequant_weight(w1q[e], w1s[e])                       # [2I, H]
        acc = X @ W1.T                                            # [n, 2I]
        h = moe.silu(acc[:, :I]) * acc[:, I:]
        hq, hs = quantize_rows(h)
        W2 = dequant_weight(w2q[e], w2s[e])                       # [H, I]
        y_pairs[slot, tok] = dequant_rows(hq, hs) @ W2.T          # [n, H]
        hq_all[pairs] = hq
        hs_all[pairs] = hs
    if return_h:
        return y_pairs, hq_all, hs_all
    return y_pairs


def combine(y_pairs: np.ndarray, topk_idx: np.ndarray, topk_w: np.ndarray) -> np.ndarray:
    """y[t] = bf16( sum over valid slots j of topk_w[t, j] * y_pairs[j, t] ), in float64.

    MonoMoe kernel design, section 1, phases 4 and 5: the weighted partials of
    a token are summed, then cast once to BF16.  Dropped pairs (index < 0)
    contribute nothing.
    """
    valid = (topk_idx >= 0).T[:, :, None]                        # [k, T, 1]
    w = topk_w.astype(np.float64).T[:, :, None]                  # [k, T, 1]
    s = np.sum(np.where(valid, w * y_pairs, 0.0), axis=0)
    return F.f64_to_bf16_bits(s)


def forward(x_bf16_bits, logits_f32, w1q, w1s, w2q, w2s, k: int, scoring: str = "softmax",
            renormalize: bool = True):
    """The whole block-FP8 layer: dict with every intermediate and y (BF16 bits [T, H])."""
    E = w1q.shape[0]
    xq, xs = quantize_act(x_bf16_bits)
    idx, w = moe.route_topk(logits_f32, k, scoring, renormalize)
    counts, offsets, perm, inv_perm = moe.permute(idx, E)
    y_pairs, hq, hs = expert_forward(xq, xs, w1q, w1s, w2q, w2s, idx, E, return_h=True)
    y = combine(y_pairs, idx, w)
    return dict(xq=xq, xs=xs, topk_idx=idx, topk_w=w, counts=counts, offsets=offsets,
                perm=perm, inv_perm=inv_perm, hq=hq, hs=hs, y_pairs=y_pairs, y=y)
