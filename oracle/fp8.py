"""FP8 (E4M3) KV pages with power-of-two scales (oracle; test infrastructure only).

vLLM-Omni RFC "Reconstruction Engine", section 3.4 (acceleration dimension 5,
quantization: "KV Cache FP8/INT8", about half the memory) and its typical
configurations table (the large-scale row: W-INT8 + KV-FP8). The pages fix
neither the FP8 format nor the scale granularity. The readings here:

  * Format: E4M3 as the OCP 8-bit floating point specification defines it (the
    "fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
    exponent field 0 holds the subnormals m * 2^-9; no infinities; the codes
    S.1111.111 are NaN; the largest finite magnitude is 1.75 * 2^8 = 448.
  * Scale granularity: one scale per stored token row, that is per (slot, head,
    K or V) group of head_dim = 64 values, which is OCP microscaling's block
    scaling with a block of 64. A page-wide scale cannot be fixed for the pages
    that fill over many frames (special pages hold 42 frames, chunk pages the
    tokens of several frames) without clipping later tokens or re-quantizing
    tokens that are already visible; a per-row scale needs neither.
  * Scale value: a power of two 2^e (an 8-bit exponent, as microscaling's E8M0
    scale), e the smallest integer with amax <= 448 * 2^e for the row's largest
    magnitude amax, clamped to [-126, 126] so that 2^e and 2^-e are normal fp32
    numbers; a row of zeros takes e = 0. A power
    of two keeps v * 2^-e exact, and dequantization decode(code) * 2^e exact in
    bf16, so quantization is the only rounding the format adds.
  * Rounding: v * 2^-e to the nearest E4M3 value, ties to the even code
    (the one whose last mantissa bit is 0); the scaled values never exceed 448,
    so no code saturates.

Functions (numpy, exact): e4m3_decode, e4m3_encode, row_exponent,
quantize_rows (bf16 bits -> codes, exponents), dequantize_rows (-> bf16 bits)
and roundtrip_rows (both). The attention over FP8 pages is the fp64 attention
of attention.py over the dequantized keys and values.
"""

import math

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """Values of E4M3 codes (uint8 array) as float64; NaN for S.1111.111."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return sign * mag


# the finite non-negative codes 0x00..0x7E, in increasing value
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = e4m3_decode(_POS_CODES)


def e4m3_encode(x):
    """Nearest E4M3 code of each float (|x| <= 448 required), ties to the even
    code. Zero keeps its sign."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    if not np.all(np.isfinite(a)) or np.any(a > E4M3_MAX):
        raise ValueError("e4m3_encode: values must be finite with magnitude <= 448")
    hi = np.searchsorted(_POS_VALUES, a, side="left")          # first value >= a
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((_POS_CODES[hi] & 1) == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    return np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)


def row_exponent(amax):
    """Scale exponent of a row with largest magnitude amax (python float):
    the smallest integer e with amax <= 448 * 2^e, clamped to [-126, 126];
    0 for amax = 0. With amax = f * 2^k, f in [0.5, 1) and 448 = 0.875 * 2^9,
    that is e = k - 9 when f <= 0.875, else k - 8."""
    if amax == 0.0:
        return 0
    f, k = math.frexp(amax)
    e = k - 9 + (1 if f > 0.875 else 0)
    return max(-126, min(126, e))


def _widen(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _narrow_exact(values):
    """float64 values that are exactly representable in bf16 -> bf16 bits."""
    f32 = np.asarray(values, dtype=np.float64).astype(np.float32)
    if not np.array_equal(f32.astype(np.float64), values):
        raise ValueError("value not representable in fp32")
    bits = f32.view(np.uint32)
    if np.any(bits & np.uint32(0xFFFF)):
        raise ValueError("value not representable in bf16")
    return (bits >> np.uint32(16)).astype(np.uint16)


def quantize_rows(bits):
    """bf16 bits [..., 64] -> (codes uint8 [..., 64], exponents int8 [...]):
    each row of head_dim values shares one power-of-two scale."""
    v = _widen(bits)
    amax = np.abs(v).max(axis=-1)
    e = np.vectorize(row_exponent, otypes=[np.int64])(amax)
    scaled = v * np.exp2(-e.astype(np.float64))[..., None]        # exact: a power of two
    return e4m3_encode(scaled), e.astype(np.int8)


def dequantize_rows(codes, exps):
    """(codes [..., 64], exponents [...]) -> bf16 bits of decode(code) * 2^e
    (exact: at most 4 significant bits)."""
    vals = e4m3_decode(codes) * np.exp2(np.asarray(exps, dtype=np.float64))[..., None]
    return _narrow_exact(vals)


def roundtrip_rows(bits):
    """bf16 bits [..., 64] -> bf16 bits of the values an FP8 page returns."""
    return dequantize_rows(*quantize_rows(bits))
