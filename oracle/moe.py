"""Plain CPU oracle of the MoE expert layer (float64 / exact integers).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import or run this module.  It shares
no code with the CUDA library and never imports it.

The layer, as the pages describe it (MegaMoE (study notes), "Baseline
implementation" and the data-flow figure after "Combine"):

    x bf16 --cast, per-32 UE8M0--> FP8 + sf
    router top-k (softmax, renormalised)         -> topk_idx, topk_w
    counting-sort permute (count -> prefix -> scatter)
    GEMM1: FP8 act x FP4 W1|W3 (per-32 UE8M0 on both) -> FP32 accumulate
        epilogue: SwiGLU (.) top-k weight -> requantise to FP8 + sf
    GEMM2: FP8 x FP4 W2 -> BF16 per (token, slot)
    combine: per token, sum of its k BF16 rows in higher precision -> BF16 y

Every floating-point step is done in float64; rounding happens only where the
pages put it (FP8/FP4 encodings, the BF16 cast of each per-pair output and of
the combined output).
"""
from __future__ import annotations

import numpy as np

from . import formats as F

GROUP = 32   # scale-group length along K (UE8M0 per 32)


# ---------------------------------------------------------------- quantisation

def quantize_act(x_bf16_bits: np.ndarray):
    """BF16 [rows, K] -> (E4M3 codes uint8 [rows, K], UE8M0 bytes uint8 [rows, K/32]).

    MegaMoE (study notes), "Dispatch" section: per token, every 32 hidden
    values share one UE8M0 scale (``per-token_cast_to_fp8, gran_k=32``).
    """
    x = F.bf16_bits_to_f64(x_bf16_bits)
    return quantize_groups_e4m3(x)


def quantize_groups_e4m3(v: np.ndarray):
    """float64 [rows, K] -> (E4M3 codes, UE8M0 bytes) with one scale per 32 along K."""
    rows, K = v.shape
    assert K % GROUP == 0
    g = v.reshape(rows, K // GROUP, GROUP)
    amax = np.max(np.abs(g), axis=-1)
    e = np.clip(F.ue8m0_exponent(amax, F.E4M3_MAX), -127, 127)
    q = np.ldexp(g, -e[..., None])                      # exact power-of-two scaling
    codes = F.encode_e4m3(q).reshape(rows, K)
    return codes, F.scale_byte(e)


def quantize_weight(w_bf16_bits: np.ndarray):
    """BF16 [G, N, K] -> (packed E2M1 uint8 [G, N, K/2], UE8M0 uint8 [G, N, K/32]).

    MegaMoE (study notes), "Expert weight quantisation" section: groups of 32
    along k, no grouping along n.  Two codes per byte, even k in the low nibble.
    """
    w = F.bf16_bits_to_f64(w_bf16_bits)
    G, N, K = w.shape
    assert K % GROUP == 0
    g = w.reshape(G, N, K // GROUP, GROUP)
    amax = np.max(np.abs(g), axis=-1)
    e = np.clip(F.ue8m0_exponent(amax, F.E2M1_MAX), -127, 127)
    q = np.ldexp(g, -e[..., None])
    codes = F.encode_e2m1(q).reshape(G, N, K)
    return F.pack_e2m1(codes), F.scale_byte(e)


def dequant_e4m3(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """E4M3 codes [..., K] with scales [..., K/32] -> float64."""
    v = F.decode_e4m3(codes)
    s = np.repeat(F.scale_value(scales), GROUP, axis=-1)
    return v * s


def dequant_e2m1(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Packed E2M1 [..., K/2] with scales [..., K/32] -> float64 [..., K]."""
    v = F.decode_e2m1(F.unpack_e2m1(packed))
    s = np.repeat(F.scale_value(scales), GROUP, axis=-1)
    return v * s


# ---------------------------------------------------------------- routing

ROUTE_SCORINGS = ("softmax", "sigmoid", "raw")


def route_topk(logits_f32: np.ndarray, k: int, scoring: str = "softmax", renormalize: bool = True):
    """Top-k routing: softmax (default) or sigmoid scores, optional renormalisation.

    MonoMoe kernel -- design, section 1 (phase 1: softmax or sigmoid top-K
    with optional renormalisation); the MegaMoE test draws ``scores = randn``
    and takes ``torch.topk`` of them, the raw scores becoming the weights
    (Counting Sort / Bucketization in DeepGEMM Mega MoE, section 7.1):
    scoring = "raw", no renormalisation.

    Selection ranks the raw logits: softmax and sigmoid are increasing, so
    the set is the same as ranking the scores, without the ties that
    rounding of the scores could create.  Equal logits: the lower expert
    index wins; output order is descending logit (lower index first on ties).

    Weights, in float64, stored as float32 (nearest even), with l_max the
    largest logit of the token and S the k selected experts:
      softmax, renormalised:  w_j = exp(l_j - l_max) / sum_{i in S} exp(l_i - l_max)
                              (the full softmax denominator cancels)
      softmax, not renorm.:   w_j = exp(l_j - l_max) / sum_{all e} exp(l_e - l_max)
      sigmoid, renormalised:  w_j = s_j / sum_{i in S} s_i,  s = 1 / (1 + exp(-l))
      sigmoid, not renorm.:   w_j = s_j
      raw (not renorm.):      w_j = l_j
    """
    if scoring not in ROUTE_SCORINGS:
        raise ValueError(f"unknown scoring {scoring!r}")
    if scoring == "raw" and renormalize:
        raise ValueError("raw scores are not renormalised")
    logits = np.asarray(logits_f32, dtype=np.float32)
    T, E = logits.shape
    assert 1 <= k <= E
    if np.any(~np.isfinite(logits)):
        raise ValueError("non-finite logit")
    idx = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float32)
    for t in range(T):
        l = logits[t].astype(np.float64)
        order = np.argsort(-l, kind="stable")       # descending value, ascending index on ties
        sel = order[:k]
        idx[t] = sel
        if scoring == "softmax":
            lmax = l[sel[0]]
            ex = np.exp(l[sel] - lmax)
            denom = ex.sum() if renormalize else np.exp(l - lmax).sum()
            wt = ex / denom
        elif scoring == "sigmoid":
            sg = 1.0 / (1.0 + np.exp(-l[sel]))
            wt = sg / sg.sum() if renormalize else sg
        else:
            wt = l[sel]
        w[t] = wt.astype(np.float32)
    return idx, w


# ---------------------------------------------------------------- counting-sort permute

def permute(topk_idx: np.ndarray, E: int):
    """Count -> prefix sum -> stable scatter of the (token, slot) pairs.

    Counting Sort / Bucketization in DeepGEMM Mega MoE, sections 2.1-2.3 and
    8.2: pair id p = token * k + slot; counts[e] = number of pairs routed to
    e; offsets = exclusive prefix of counts (E + 1 entries); the pairs of
    expert e occupy perm[offsets[e] : offsets[e + 1]].  The pages take the
    slot inside an expert from an atomic counter (order not fixed); here it is
    the rank of p among that expert's pairs (stable, token-ascending).
    A negative index marks a dropped pair (section 7.1 listing): it is not
    counted and gets inv_perm = -1.
    """
    flat = np.asarray(topk_idx, dtype=np.int64).reshape(-1)
    P = flat.size
    if np.any(flat >= E):
        raise ValueError("expert index out of range")
    counts = np.zeros(E, dtype=np.int64)
    for e in flat[flat >= 0]:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.zeros(int(offsets[E]), dtype=np.int64)
    for e in range(E):
        pairs_of_e = np.nonzero(flat == e)[0]        # ascending pair ids
        perm[offsets[e]:offsets[e + 1]] = pairs_of_e
    inv_perm = np.full(P, -1, dtype=np.int64)
    inv_perm[perm] = np.arange(perm.size)
    return (counts.astype(np.int32), offsets.astype(np.int32),
            perm.astype(np.int32), inv_perm.astype(np.int32))


# ---------------------------------------------------------------- expert GEMMs

def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def expert_forward(xq, xs, w1q, w1s, w2q, w2s, topk_idx, topk_w, E: int,
                   experts=None, return_h: bool = False):
    """GEMM1 + SwiGLU (.) weight + FP8 requantisation + GEMM2 for every pair.

    Weights are in the natural layout: l1 [E, 2I, H] with gate rows [0, I)
    and up rows [I, 2I) (MegaMoE (study notes), "Original weight layout"),
    l2 [E, H, I].  For a pair p = (t, j) routed to expert e:

        acc   = deq(xq[t]) . deq(W1[e])^T                      (2I values)
        h     = silu(acc[:I]) * acc[I:] * topk_w[t, j]         (I values)
        hq,hs = E4M3 + UE8M0 per 32 of h                       (L1 epilogue)
        y_p   = bf16( deq(hq, hs) . deq(W2[e])^T )             (H values)

    (Warp Specialization: DeepEP vs Mega MoE, L1 and L2 epilogue listings;
    MegaMoE (study notes), "L1 epilogue" and "L2 epilogue".)  The top-k
    weight multiplies h before requantisation.

    Returns y_pairs as BF16 bits [k, T, H] (rows of dropped pairs are 0) and,
    with ``return_h``, hq [P, I] / hs [P, I/32] indexed by pair id.
    ``experts`` restricts the work to a subset of experts (other rows 0).
    """
    T, k = topk_idx.shape
    H = xq.shape[1]
    I = w2q.shape[2] * 2
    y_pairs = np.zeros((k, T, H), dtype=np.uint16)
    hq_all = np.zeros((T * k, I), dtype=np.uint8)
    hs_all = np.zeros((T * k, I // GROUP), dtype=np.uint8)
    flat = topk_idx.reshape(-1)
    todo = range(E) if experts is None else experts
    for e in todo:
        pairs = np.nonzero(flat == e)[0]
        if pairs.size == 0:
            continue
        tok = pairs // k
        slot = pairs % k
        X = dequant_e4m3(xq[tok], xs[tok])                       # [n, H]
        W1 = dequant_e2m1(w1q[e], w1s[e])                        # [2I, H]
        acc = X @ W1.T                                           # [n, 2I]
        gate, up = acc[:, :I], acc[:, I:]
        wts = topk_w[tok, slot].astype(np.float64)
        h = silu(gate) * up * wts[:, None]
        hq, hs = quantize_groups_e4m3(h)
        Hd = dequant_e4m3(hq, hs)                                # [n, I]
        W2 = dequant_e2m1(w2q[e], w2s[e])                        # [H, I]
        y = Hd @ W2.T                                            # [n, H]
        y_pairs[slot, tok] = F.f64_to_bf16_bits(y)
        hq_all[pairs] = hq
        hs_all[pairs] = hs
    if return_h:
        return y_pairs, hq_all, hs_all
    return y_pairs


def combine(y_pairs: np.ndarray, topk_idx: np.ndarray) -> np.ndarray:
    """y[t] = bf16( sum over valid slots j of y_pairs[j, t] ), summed in float64.

    MegaMoE (study notes), "Combine" and "L2 epilogue": the per-pair outputs
    stay BF16 and the k copies of a token are summed in higher precision, then
    cast to BF16.  The top-k weight was already applied before GEMM2, so the
    sum is unweighted.  Dropped pairs (index < 0) contribute nothing.
    """
    k, T, H = y_pairs.shape
    vals = F.bf16_bits_to_f64(y_pairs)                          # [k, T, H]
    valid = (topk_idx >= 0).T[:, :, None]                       # [k, T, 1]
    s = np.sum(np.where(valid, vals, 0.0), axis=0)
    return F.f64_to_bf16_bits(s)


def forward(x_bf16_bits, logits_f32, w1q, w1s, w2q, w2s, k: int, scoring: str = "softmax",
            renormalize: bool = True):
    """The whole layer: returns dict with every intermediate and y (BF16 bits [T, H])."""
    E = w1q.shape[0]
    xq, xs = quantize_act(x_bf16_bits)
    idx, w = route_topk(logits_f32, k, scoring, renormalize)
    counts, offsets, perm, inv_perm = permute(idx, E)
    y_pairs, hq, hs = expert_forward(xq, xs, w1q, w1s, w2q, w2s, idx, w, E, return_h=True)
    y = combine(y_pairs, idx)
    return dict(xq=xq, xs=xs, topk_idx=idx, topk_w=w, counts=counts, offsets=offsets,
                perm=perm, inv_perm=inv_perm, hq=hq, hs=hs, y_pairs=y_pairs, y=y)
