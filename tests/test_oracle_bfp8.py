"""Pins for the block-FP8 oracle (CPU only).

The variant is the single-kernel MoE of the MonoMoe kernel design page
("Fixed shape", section 1): E4M3 weights with 128 x 128 block scales, FP8
activations with per-token scales per 128 values, FP32 down-projection
partials weighted and summed per token.  Each pin reaches the oracle's result
by another route: hand-computed encodings (tests/golden/bfp8_act_quant.txt),
PyTorch's own float8_e4m3fn cast, error bounds, invariances, and the expert
GEMMs rewritten per 128-wide K block in exact integer arithmetic (the
formulation the kernels use) instead of dequantise-then-matmul.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import bfp8 as B
from oracle import formats as F
from oracle import moe as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _value(s: str) -> float:
    s = s.strip()
    if "*2^" in s:
        a, n = s.split("*2^")
        return float(Fraction(a)) * 2.0 ** int(n)
    return float(Fraction(s))


def _torch_e4m3(q32: np.ndarray) -> np.ndarray:
    """PyTorch's float32 -> float8_e4m3fn cast (nearest-even), as code bytes."""
    t = torch.from_numpy(np.ascontiguousarray(q32, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


# ---------------------------------------------------------------- activation cast

def test_golden_activation_groups():
    n = 0
    with open(os.path.join(GOLDEN, "bfp8_act_quant.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            scale_hex, codes_txt = rhs.split(";")
            row = np.zeros((1, 128), np.float64)
            idx = []
            for tok in lhs.split():
                i, v = tok.split(":")
                row[0, int(i)] = _value(v)
                idx.append(int(i))
            codes, s = B.quantize_rows(row)
            assert s.dtype == np.float32 and s.shape == (1, 1)
            assert int(s.view(np.uint32)[0, 0]) == int(scale_hex, 16), line
            want = [int(c, 16) for c in codes_txt.split()]
            assert [int(codes[0, i]) for i in idx] == want, line
            rest = np.ones(128, bool)
            rest[idx] = False
            assert np.all(codes[0, rest] == 0), line
            n += 1
    assert n == 5


def _random_rows(rows, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, K, generator=g)
    # magnitudes from 2^-30 to 2^30 across groups, plus an all-zero group
    mag = torch.exp2(torch.randint(-30, 31, (rows, K // 128, 1), generator=g).float())
    x = (x.view(rows, K // 128, 128) * mag).view(rows, K)
    x[0, :128] = 0.0
    return _bits(x)


def test_activation_codes_match_library_cast():
    """Given the scale, the codes are PyTorch's own E4M3 cast of value / scale."""
    x = _random_rows(16, 1024, seed=5)
    codes, s = B.quantize_act(x)
    v32 = F.bf16_bits_to_f64(x).astype(np.float32).reshape(16, 8, 128)
    nz = s > 0
    q32 = v32 / np.where(nz, s, np.float32(1))[..., None]
    want = np.where(nz[..., None], _torch_e4m3(q32), 0).reshape(16, 1024)
    assert np.array_equal(codes, want)


def test_activation_amax_element_lands_on_448_and_error_bound():
    x = _random_rows(8, 512, seed=6)
    codes, s = B.quantize_act(x)
    v = F.bf16_bits_to_f64(x).reshape(8, 4, 128)
    c = codes.reshape(8, 4, 128)
    for r in range(8):
        for g in range(4):
            a = np.abs(v[r, g])
            if a.max() == 0:
                assert s[r, g] == 0 and np.all(c[r, g] == 0)
                continue
            i = int(np.argmax(a))
            assert c[r, g, i] & 0x7F == 0x7E           # |code| = 448
            # dequantised error: half an E4M3 step at the value's binade
            # (subnormal step 2^-9 below 2^-6), times the scale, plus float32 slack
            d = F.decode_e4m3(c[r, g]) * np.float64(s[r, g])
            q = a / np.float64(s[r, g])
            step = np.where(q < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(q, 2.0 ** -6))) - 3))
            assert np.all(np.abs(d - v[r, g]) <= (0.5 * step * (1 + 2.0 ** -20) + 2.0 ** -22 * q) * s[r, g])


def test_activation_scaling_by_power_of_two():
    x = _random_rows(4, 256, seed=7)
    xf = F.bf16_bits_to_f64(x)
    c0, s0 = B.quantize_rows(xf)
    for n in (-5, 3):
        c1, s1 = B.quantize_rows(np.ldexp(xf, n))
        assert np.array_equal(c0, c1)
        assert np.array_equal(s1, np.ldexp(s0, n).astype(np.float32))


# ---------------------------------------------------------------- weight cast

def test_weight_block_hand_case():
    """One 256 x 256 matrix, four 128 x 128 blocks, written out by hand.

    Block (0,0): amax 896 -> scale 2; -896 -> -448 (0xfe), 6 -> 3 (0x44).
    Block (0,1): all zero -> scale 0.  Block (1,0): 448 -> scale 1,
    0.75 = 1.5 * 2^-1 -> exponent field 6, mantissa 100b -> 0x34.  Block (1,1): amax 1 -> scale fl32(1/448).
    """
    w = np.zeros((1, 256, 256), np.float32)
    w[0, 0, 0] = -896.0
    w[0, 5, 7] = 6.0
    w[0, 200, 3] = 448.0
    w[0, 130, 100] = 0.75
    w[0, 255, 255] = 1.0
    codes, s = B.quantize_weight(_bits(torch.from_numpy(w)))
    assert s.shape == (1, 2, 2) and s.dtype == np.float32
    assert s[0, 0, 0] == 2.0 and s[0, 0, 1] == 0.0 and s[0, 1, 0] == 1.0
    assert int(s[0, 1, 1:2].view(np.uint32)[0]) == 0x3B124925
    assert codes[0, 0, 0] == 0xFE and codes[0, 5, 7] == 0x44
    assert codes[0, 200, 3] == 0x7E and codes[0, 130, 100] == 0x34 and codes[0, 255, 255] == 0x7E
    assert np.count_nonzero(codes) == 5


def test_weight_codes_match_library_cast_and_blocks_are_local():
    g = torch.Generator().manual_seed(8)
    w = torch.randn(2, 256, 384, generator=g) * 0.02
    wb = _bits(w)
    codes, s = B.quantize_weight(wb)
    w32 = F.bf16_bits_to_f64(wb).astype(np.float32)
    sfull = np.repeat(np.repeat(s, 128, axis=1), 128, axis=2)
    assert np.array_equal(codes, _torch_e4m3(w32 / sfull))
    # every block's largest magnitude encodes to +-448
    for gi in range(2):
        for nb in range(2):
            for kb in range(3):
                blk = np.abs(w32[gi, nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128])
                r, c = np.unravel_index(int(np.argmax(blk)), blk.shape)
                assert codes[gi, nb * 128 + r, kb * 128 + c] & 0x7F == 0x7E
    # scaling one block by 2^4 moves only that block's scale, no code
    w2 = w.clone()
    w2[1, 128:256, 128:256] *= 16.0
    codes2, s2 = B.quantize_weight(_bits(w2))
    assert np.array_equal(codes, codes2)
    want = s.copy()
    want[1, 1, 1] *= 16
    assert np.array_equal(s2, want)


# ---------------------------------------------------------------- the layer

def _layer(T, H, I, E, seed, sigma=0.05):
    g = torch.Generator().manual_seed(seed)
    x = _bits(torch.randn(T, H, generator=g))
    logits = torch.randn(T, E, generator=g).numpy()
    l1 = _bits(torch.randn(E, 2 * I, H, generator=g) * sigma)
    l2 = _bits(torch.randn(E, H, I, generator=g) * sigma)
    # different magnitudes per 128-row block, so a transposed block index shows
    l1 = _bits(torch.from_numpy(F.bf16_bits_to_f64(l1)).float()
               * torch.exp2(torch.randint(-2, 3, (E, 2 * I // 128, 1, 1), generator=g).float())
               .expand(E, 2 * I // 128, 128, 1).reshape(E, 2 * I, 1))
    w1q, w1s = B.quantize_weight(l1)
    w2q, w2s = B.quantize_weight(l2)
    return x, logits, w1q, w1s, w2q, w2s


def _int_code(c: np.ndarray) -> np.ndarray:
    """E4M3 codes as exact integers: value * 2^9 (every E4M3 value is a multiple of 2^-9)."""
    return np.rint(F.decode_e4m3(c) * 512.0).astype(np.int64)


def _gemm_per_kblock(aq, as_, wq, ws):
    """out[n, j] = sum over 128-wide K blocks kb of ws[j/128, kb] * as_[n, kb] * <a_n, w_j>_kb.

    Integer dot products per K block (codes as multiples of 2^-9), then the
    two float32 scales of the block: the kernels' formulation, written
    without the oracle's dequantise-then-matmul.
    """
    n, K = aq.shape
    J = wq.shape[0]
    ai = _int_code(aq).reshape(n, K // 128, 128)
    wi = _int_code(wq).reshape(J, K // 128, 128)
    dots = np.einsum("nbk,jbk->njb", ai, wi).astype(np.float64) * 2.0 ** -18   # exact
    sw = np.repeat(ws.astype(np.float64), 128, axis=0)                        # [J, K/128]
    return np.einsum("njb,jb,nb->nj", dots, sw, as_.astype(np.float64))


def _dense_expert(xq, xs, w1q, w1s, w2q, w2s, I):
    """One expert as a dense MLP on quantised operands, in the per-K-block form."""
    acc = _gemm_per_kblock(xq, xs, w1q, w1s)
    gate, up = acc[:, :I], acc[:, I:]
    h = gate / (1.0 + np.exp(-gate)) * up
    hq, hs = B.quantize_rows(h)
    return _gemm_per_kblock(hq, hs, w2q, w2s), hq, hs


def test_single_expert_equals_dense_mlp():
    T, H, I = 12, 256, 256
    x, logits, w1q, w1s, w2q, w2s = _layer(T, H, I, 1, seed=9)
    out = B.forward(x, logits, w1q, w1s, w2q, w2s, k=1)
    assert np.all(out["topk_w"] == 1.0)
    y, hq, hs = _dense_expert(out["xq"], out["xs"], w1q[0], w1s[0], w2q[0], w2s[0], I)
    assert np.array_equal(out["hq"], hq) and np.array_equal(out["hs"], hs)
    assert np.array_equal(out["y"], F.f64_to_bf16_bits(y))


@pytest.mark.parametrize("E,k,seed", [(2, 2, 10), (3, 2, 11), (4, 3, 12)])
def test_weighted_sum_of_dense_experts(E, k, seed):
    """Every token: y = bf16( sum over its k experts of w_j * dense_expert_j(token) )."""
    T, H, I = 10, 256, 128
    x, logits, w1q, w1s, w2q, w2s = _layer(T, H, I, E, seed=seed)
    out = B.forward(x, logits, w1q, w1s, w2q, w2s, k=k)
    dense = [_dense_expert(out["xq"], out["xs"], w1q[e], w1s[e], w2q[e], w2s[e], I)[0] for e in range(E)]
    y = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            y[t] += np.float64(out["topk_w"][t, j]) * dense[out["topk_idx"][t, j]][t]
    assert np.array_equal(out["y"], F.f64_to_bf16_bits(y))


def test_zero_input_gives_zero_output():
    T, H, I, E, k = 6, 128, 128, 4, 2
    _, logits, w1q, w1s, w2q, w2s = _layer(T, H, I, E, seed=13)
    out = B.forward(np.zeros((T, H), np.uint16), logits, w1q, w1s, w2q, w2s, k=k)
    assert np.all(out["y"] == 0) and np.all(out["hq"] == 0) and np.all(out["hs"] == 0)
    assert np.all(out["xs"] == 0)


def test_relabelling_experts_leaves_output_unchanged():
    T, H, I, E, k = 9, 128, 128, 5, 2
    x, logits, w1q, w1s, w2q, w2s = _layer(T, H, I, E, seed=14)
    out = B.forward(x, logits, w1q, w1s, w2q, w2s, k=k)
    sg = np.array([3, 0, 4, 1, 2])
    out2 = B.forward(x, logits[:, sg], w1q[sg], w1s[sg], w2q[sg], w2s[sg], k=k)
    assert np.array_equal(out["y"], out2["y"])
    assert np.array_equal(out["y_pairs"], out2["y_pairs"])


def test_combine_weights_each_pair_once_and_skips_dropped():
    """Hand case: 1.0 * 0.25 + 3.0 * 0.75 = 2.5 (BF16 0x4020); a dropped slot adds nothing."""
    y_pairs = np.array([[[1.0]], [[3.0]], [[100.0]]])        # [k=3, T=1, H=1]
    idx = np.array([[0, 1, -1]])
    w = np.array([[0.25, 0.75, 0.5]], np.float32)
    assert B.combine(y_pairs, idx, w)[0, 0] == 0x4020


def test_routing_and_permute_are_the_layers_own():
    T, H, I, E, k = 7, 128, 128, 6, 3
    x, logits, w1q, w1s, w2q, w2s = _layer(T, H, I, E, seed=15)
    for scoring, renorm in (("softmax", True), ("sigmoid", False)):
        out = B.forward(x, logits, w1q, w1s, w2q, w2s, k=k, scoring=scoring, renormalize=renorm)
        idx, w = O.route_topk(logits, k, scoring, renorm)
        assert np.array_equal(out["topk_idx"], idx) and np.array_equal(out["topk_w"], w)
        c, o, p, ip = O.permute(idx, E)
        assert np.array_equal(out["perm"], p) and np.array_equal(out["offsets"], o)
