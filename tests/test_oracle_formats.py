"""Pins for the oracle's number formats (CPU only).

Each check compares the oracle with something written independently of it:
hand tables in tests/golden, brute force over every code, exact rational
arithmetic, or torch's own float32 -> bfloat16 cast.
"""
import math
import os
import re
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import moe as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_value(s: str) -> float:
    s = s.strip()
    neg = s.startswith("-")
    if neg:
        s = s[1:]
    m = re.fullmatch(r"(\d+)\*2\^(-?\d+)", s)
    if m:
        v = math.ldexp(float(m.group(1)), int(m.group(2)))
    elif "/" in s:
        a, b = s.split("/")
        v = float(Fraction(int(a), int(b)))
    else:
        v = float(int(s))
    return -v if neg else v


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            rows.append((lhs.strip(), int(rhs.strip(), 0)))
    return rows


@pytest.mark.parametrize("fname,enc", [("e2m1_encode.txt", F.encode_e2m1),
                                       ("e4m3_encode.txt", F.encode_e4m3)])
def test_golden_encodings(fname, enc):
    for lhs, want in _golden(fname):
        v = _parse_value(lhs)
        got = int(enc(np.array([v]))[0])
        assert got == want, f"{fname}: {lhs} -> {got:#x}, expected {want:#x}"


def test_golden_ue8m0():
    for lhs, want in _golden("ue8m0.txt"):
        fmt, val = lhs.split()
        q = F.E4M3_MAX if fmt == "e4m3" else F.E2M1_MAX
        e = F.ue8m0_exponent(np.array([_parse_value(val)]), q)
        assert int(F.scale_byte(e)[0]) == want, lhs


def _brute_exponent(amax: float, qmax: int) -> int:
    """Smallest integer e with qmax * 2**e >= amax, by exact rational search."""
    a = Fraction(amax)
    e = 0
    while Fraction(qmax) * Fraction(2) ** e < a:
        e += 1
    while Fraction(qmax) * Fraction(2) ** (e - 1) >= a:
        e -= 1
    return e


def test_ue8m0_matches_exact_definition():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        np.abs(rng.standard_normal(400)) * 10.0 ** rng.integers(-6, 6, 400),
        [448.0, 448.0 * (1 + 2 ** -7), 6.0, 6.0 * (1 + 2 ** -52), 0.875, 0.75, 2.0 ** -30,
         np.nextafter(448.0, 0), np.nextafter(6.0, 0)],
    ])
    for q in (448, 6):
        got = F.ue8m0_exponent(vals, float(q))
        for v, g in zip(vals, got):
            assert g == _brute_exponent(float(v), q), (q, v)


def _brute_encode(v: float, mags: np.ndarray, sign_bit: int) -> int:
    """Nearest code by scanning every code; ties to the code with LSB 0."""
    a = abs(v)
    best, best_d = None, None
    for code, m in enumerate(mags):
        d = abs(Fraction(a) - Fraction(float(m)))
        if best is None or d < best_d or (d == best_d and code % 2 == 0):
            best, best_d = code, d
    return best | (sign_bit if math.copysign(1.0, v) < 0 else 0)


@pytest.mark.parametrize("mags,sign,enc", [(F.E4M3_MAGS, 0x80, F.encode_e4m3),
                                           (F.E2M1_MAGS, 0x8, F.encode_e2m1)])
def test_encode_matches_brute_force(mags, sign, enc):
    rng = np.random.default_rng(11)
    mids = (mags[1:] + mags[:-1]) / 2                      # every tie point
    vals = np.concatenate([rng.uniform(-mags[-1], mags[-1], 300), mids, -mids, mags, -mags])
    got = enc(vals)
    for v, g in zip(vals, got):
        assert int(g) == _brute_encode(float(v), mags, sign), v


def test_decode_encode_identity_all_codes():
    c8 = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(F.encode_e4m3(F.decode_e4m3(c8)), c8)
    c4 = np.arange(16, dtype=np.uint8)
    assert np.array_equal(F.encode_e2m1(F.decode_e2m1(c4)), c4)
    # the tables themselves: E4M3 top value, E2M1 list
    assert F.E4M3_MAGS[-1] == 448.0 and F.E4M3_MAGS[1] == 2.0 ** -9
    assert list(F.E2M1_MAGS) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_pack_nibble_order():
    codes = np.array([[1, 2, 3, 0xF]], dtype=np.uint8)
    assert F.pack_e2m1(codes).tolist() == [[0x21, 0xF3]]
    assert np.array_equal(F.unpack_e2m1(F.pack_e2m1(codes)), codes)


def test_bf16_rounding_matches_torch_on_float32_values():
    rng = np.random.default_rng(3)
    v32 = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    v32 = np.concatenate([v32, np.array([1e-40, -3e-39, 0.0, -0.0], np.float32)])
    want = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = F.f64_to_bf16_bits(v32.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_rounding_is_single_step():
    # 1 + 2^-8 + 2^-30: nearest BF16 is 1 + 2^-7; a float32 detour would tie back to 1.0
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert F.bf16_bits_to_f64(F.f64_to_bf16_bits(np.array([v])))[0] == 1.0 + 2.0 ** -7
    assert F.bf16_bits_to_f64(F.f64_to_bf16_bits(np.array([1.0 + 2.0 ** -8])))[0] == 1.0


def test_quantize_act_hand_group():
    # one group of 32: amax 3.0 -> e = ceil(log2(3/448)) = -7, q = v * 128
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0] = 3.0
    x[0, 1] = -1.0
    x[0, 2] = 2.0 ** -20
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    codes, scales = O.quantize_act(bits)
    assert scales.tolist() == [[127 - 7]]
    assert codes[0, 0] == F.encode_e4m3(np.array([384.0]))[0] == 0x7C
    assert codes[0, 1] == 0x80 | 0x70          # -128 = -(1.0 * 2^7): E = 14, m = 0
    assert codes[0, 2] == 0x00                 # 2^-13 underflows to +0
    assert np.all(codes[0, 3:] == 0)


def test_quantize_scale_invariance():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 128)).astype(np.float32)
    b0 = torch.from_numpy(x).to(torch.bfloat16)
    for n in (-5, 3):
        b1 = (b0.float() * 2.0 ** n).to(torch.bfloat16)     # exact: power-of-two scaling
        c0, s0 = O.quantize_act(b0.view(torch.int16).numpy().view(np.uint16))
        c1, s1 = O.quantize_act(b1.view(torch.int16).numpy().view(np.uint16))
        assert np.array_equal(c0, c1)
        assert np.array_equal(s1.astype(int), s0.astype(int) + n)


def test_quantize_weight_roundtrip_error_bound():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((2, 8, 64)) * 0.02).astype(np.float32)
    bits = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q, s = O.quantize_weight(bits)
    assert q.shape == (2, 8, 32) and s.shape == (2, 8, 2)
    wd = O.dequant_e2m1(q, s)
    wf = F.bf16_bits_to_f64(bits)
    # E2M1 error <= half the widest gap (2 between 4 and 6 -> 1) times the scale
    scale = np.repeat(F.scale_value(s), 32, axis=-1)
    assert np.all(np.abs(wd - wf) <= 1.0 * scale)
    # the group maximum is representable to within the top gap and never clipped
    g = np.abs(wf).reshape(2, 8, 2, 32).max(-1)
    assert np.all(g <= 6.0 * F.scale_value(s))
    assert np.all(g > 3.0 * F.scale_value(s))   # e is the smallest exponent that fits
