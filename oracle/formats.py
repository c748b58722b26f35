"""Number formats of the MoE expert layer, written out from their definitions.

TEST INFRASTRUCTURE ONLY.  This module is part of the CPU oracle.  Only the
test-suite, the smoke check of ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may import it; the CUDA product path never does.

Formats (all arithmetic in float64 / exact integer arithmetic):

* FP8 E4M3 ("FN" variant: no infinities, max finite 448) -- the activation
  format.  MegaMoE (study notes), "Dispatch" and "GEMM" sections: tokens are
  cast to FP8 with one UE8M0 scale per 32 values along hidden.
* FP4 E2M1 (values 0, 0.5, 1, 1.5, 2, 3, 4, 6) -- the weight format.  MegaMoE
  (study notes), "Expert weight quantisation" section: a BF16 [G, n, k] matrix
  becomes FP4 [G, n, k] plus UE8M0 [G, n, k/32], no grouping along n.
* UE8M0 -- an 8-bit biased power-of-two exponent, byte = e + 127.
  The scale rule is 2**ceil(log2(amax / Q)) with Q = 448 (E4M3) or 6 (E2M1);
  the pages name the helper (``get_e4m3_sf_and_sf_inv``, Warp Specialization:
  DeepEP vs Mega MoE, L1 epilogue listing) but do not print it, so the rule
  is the one the layer's specification fixes.
* BF16 with round-to-nearest-even from an exact float64 value.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0


def _e4m3_magnitudes() -> np.ndarray:
    """Magnitude of every non-NaN E4M3 code 0..126 (sign bit clear)."""
    mags = np.zeros(127, dtype=np.float64)
    for code in range(127):
        exp_field = code >> 3
        man = code & 7
        if exp_field == 0:                      # subnormal: man/8 * 2^-6
            mags[code] = man * 2.0 ** -9
        else:                                   # normal: (1 + man/8) * 2^(E-7)
            mags[code] = (1.0 + man / 8.0) * 2.0 ** (exp_field - 7)
    return mags


def _e2m1_magnitudes() -> np.ndarray:
    """Magnitude of the 8 E2M1 codes 0..7 (sign bit clear)."""
    mags = np.zeros(8, dtype=np.float64)
    for code in range(8):
        exp_field = code >> 1
        man = code & 1
        if exp_field == 0:                      # subnormal: man * 0.5
            mags[code] = man * 0.5
        else:                                   # (1 + man/2) * 2^(E-1)
            mags[code] = (1.0 + man / 2.0) * 2.0 ** (exp_field - 1)
    return mags


E4M3_MAGS = _e4m3_magnitudes()   # strictly increasing, last = 448
E2M1_MAGS = _e2m1_magnitudes()   # [0, .5, 1, 1.5, 2, 3, 4, 6]
E4M3_SIGN = 0x80
E2M1_SIGN = 0x8


def ue8m0_exponent(amax: np.ndarray, qmax: float) -> np.ndarray:
    """Smallest integer e with qmax * 2**e >= amax, evaluated exactly.

    With amax = m * 2**f (frexp, m in [0.5, 1)) and qmax = c * 2**b
    (c in [0.5, 1)): e = f - b when m <= c, else f - b + 1.  amax == 0 gives
    -inf in the definition; it is returned as -127 (the clamp below).
    """
    amax = np.asarray(amax, dtype=np.float64)
    if np.any(~np.isfinite(amax)) or np.any(amax < 0):
        raise ValueError("amax must be finite and non-negative")
    c, b = np.frexp(qmax)
    m, f = np.frexp(amax)
    e = np.where(m <= c, f - b, f - b + 1).astype(np.int64)
    return np.where(amax == 0, -127, e)


def scale_byte(e: np.ndarray) -> np.ndarray:
    """UE8M0 byte for exponent e: e + 127 clamped to [0, 254] (255 = NaN is never produced)."""
    return np.clip(np.asarray(e, dtype=np.int64) + 127, 0, 254).astype(np.uint8)


def _encode_rne(q: np.ndarray, mags: np.ndarray, sign_bit: int) -> np.ndarray:
    """Round |q| to the nearest magnitude in ``mags``; ties go to the even code."""
    q = np.asarray(q, dtype=np.float64)
    if np.any(~np.isfinite(q)):
        raise ValueError("non-finite value reached the encoder")
    a = np.abs(q)
    if np.any(a > mags[-1]):
        raise ValueError("value above the format's largest finite magnitude")
    hi = np.searchsorted(mags, a, side="left")          # first mag >= a
    hi = np.minimum(hi, len(mags) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - mags[lo]
    d_hi = mags[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a == mags[hi], hi, code)            # exact hits
    neg = np.signbit(q)                                 # keeps the sign of -0 and of values rounding to 0
    return (code | np.where(neg, sign_bit, 0)).astype(np.uint8)


def encode_e4m3(q: np.ndarray) -> np.ndarray:
    return _encode_rne(q, E4M3_MAGS, E4M3_SIGN)


def encode_e2m1(q: np.ndarray) -> np.ndarray:
    return _encode_rne(q, E2M1_MAGS, E2M1_SIGN)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.int64)
    mag_code = codes & 0x7F
    if np.any(mag_code == 0x7F):
        raise ValueError("E4M3 NaN code")
    v = E4M3_MAGS[mag_code]
    return np.where(codes & 0x80, -v, v)


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.int64)
    v = E2M1_MAGS[codes & 0x7]
    return np.where(codes & 0x8, -v, v)


def scale_value(byte: np.ndarray) -> np.ndarray:
    """2**(byte - 127) as float64."""
    return np.ldexp(1.0, np.asarray(byte, dtype=np.int64) - 127)


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Two E2M1 codes per byte along the last axis: even index in the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    assert codes.shape[-1] % 2 == 0
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


# ---------------------------------------------------------------- BF16

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of BF16 bit patterns (uint16) as float64."""
    bits = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 values to BF16 (nearest, ties to even) in one step.

    BF16 keeps 8 significant bits; below 2**-126 the spacing is 2**-133
    (subnormals).  Rounding straight from float64 avoids the double rounding
    of a float64 -> float32 -> bf16 chain.
    """
    v = np.asarray(v, dtype=np.float64)
    if np.any(~np.isfinite(v)):
        raise ValueError("non-finite value")
    _, ex = np.frexp(v)                       # v = m * 2**ex, m in [0.5, 1)
    quantum = np.maximum(ex - 8, -133)        # exponent of the last kept bit
    r = np.ldexp(np.rint(np.ldexp(v, -quantum)), quantum)   # rint = ties to even
    r = np.where(v == 0, v, r)                # keep signed zeros
    if np.any(np.abs(r) > 3.3895313892515355e38):
        raise ValueError("BF16 overflow")
    bits = r.astype(np.float32).view(np.uint32) >> 16   # r is exact in float32
    return bits.astype(np.uint16)
