"""Pins of the FP8 (E4M3) page oracle against what does not depend on it: the
library's own float8_e4m3fn type (PyTorch's implementation of the OCP E4M3
format) for every code and for rounding, and the closed-form properties of the
power-of-two row scale (minimality, the error bound of round-to-nearest)."""

import numpy as np
import pytest
import torch

from oracle.fp8 import (e4m3_decode, e4m3_encode, dequantize_rows, quantize_rows, roundtrip_rows,
                        row_exponent)


def _torch_decode(codes):
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _torch_encode(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_decode_matches_the_library_type_for_all_256_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours, lib = e4m3_decode(codes), _torch_decode(codes)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    assert np.isnan(ours).sum() == 2                                  # 0x7F and 0xFF only
    ok = ~np.isnan(lib)
    assert np.array_equal(ours[ok], lib[ok])
    # landmarks of the format: largest finite, smallest normal and subnormal, one
    assert e4m3_decode([0x7E, 0x08, 0x01, 0x38, 0xB8]).tolist() == [448.0, 2.0 ** -6, 2.0 ** -9,
                                                                       1.0, -1.0]


def test_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    back = e4m3_encode(e4m3_decode(codes))
    # +0 and -0 keep their sign bit; every other code round-trips exactly
    assert np.array_equal(back, codes)


def test_encode_ties_go_to_the_even_code():
    pos = e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2                                   # exact in float64
    ours = e4m3_encode(mids)
    assert np.all((ours & 1) == 0)
    assert np.array_equal(ours, _torch_encode(mids))                  # midpoints are exact in fp32
    assert np.array_equal(e4m3_encode(-mids), _torch_encode(-mids))


def test_encode_matches_the_library_rounding_on_random_values():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.uniform(-448, 448, 20000),
                        rng.normal(0, 1, 20000),
                        rng.uniform(-2.0 ** -6, 2.0 ** -6, 20000),          # subnormal range
                        np.ldexp(rng.uniform(1, 2, 2000), rng.integers(-12, 8, 2000))])
    x = x.astype(np.float32).astype(np.float64)                      # values the kernel sees
    assert np.array_equal(e4m3_encode(x), _torch_encode(x))
    with pytest.raises(ValueError):
        e4m3_encode([449.0])


@pytest.mark.parametrize("amax", [1.0, 448.0, 449.0, 224.0, 224.0 * (1 + 2 ** -20), 3.5, 2.0 ** -40,
                                  1e-3, 7.0, 7.0000001, 65504.0, 1e30])
def test_row_exponent_is_the_smallest_that_fits(amax):
    e = row_exponent(amax)
    assert amax <= 448.0 * 2.0 ** e
    assert amax > 448.0 * 2.0 ** (e - 1)


def test_row_exponent_edges():
    assert row_exponent(0.0) == 0
    assert row_exponent(1e-60) == -126                               # clamped below
    assert row_exponent(448.0 * 2.0 ** 127) == 126
    rng = np.random.default_rng(3)
    for amax in np.ldexp(rng.uniform(0.5, 1, 500), rng.integers(-100, 100, 500)):
        e = row_exponent(float(amax))
        assert amax <= 448.0 * 2.0 ** e and amax > 448.0 * 2.0 ** (e - 1)


def _bf16_bits(x):
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16                          # round to nearest even
    return u.astype(np.uint16)


def _from_bits(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_quantized_rows_are_within_half_a_step():
    rng = np.random.default_rng(11)
    rows = np.concatenate([rng.normal(0, 1, (300, 64)), rng.normal(0, 1e-3, (100, 64)),
                           rng.normal(0, 300, (100, 64)), np.zeros((2, 64))])
    rows[5, 7] = 0.0
    bits = _bf16_bits(rows)
    v = _from_bits(bits)
    codes, exps = quantize_rows(bits)
    deq = _from_bits(dequantize_rows(codes, exps))
    assert np.array_equal(deq, _from_bits(roundtrip_rows(bits)))
    amax = np.abs(v).max(axis=1)
    scaled_max = amax * np.exp2(-exps.astype(np.float64))
    nz = amax > 0
    assert np.all(scaled_max[nz] <= 448) and np.all(scaled_max[nz] > 224)
    s = np.abs(v) * np.exp2(-exps.astype(np.float64))[:, None]
    # half the E4M3 spacing at each scaled magnitude: 2^(floor(log2 s) - 4) for
    # normals (s >= 2^-6), 2^-10 for subnormals
    half = np.where(s >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(s, 2.0 ** -6))) - 4), 2.0 ** -10)
    err = np.abs(deq - v) * np.exp2(-exps.astype(np.float64))[:, None]
    assert np.all(err <= half)
    assert np.array_equal(deq[-2:], np.zeros((2, 64)))                # zero rows stay zero
    assert np.signbit(deq[v == 0]).sum() == np.signbit(v[v == 0]).sum()


def test_a_planted_scale_error_is_caught():
    """An exponent one too small leaves row maxima past 448, which no code holds
    (the encoder refuses them); one too large breaks minimality (the scaled row
    maximum drops to 224 or below, wasting the top binade)."""
    rng = np.random.default_rng(5)
    v = _from_bits(_bf16_bits(rng.normal(0, 1, (50, 64))))
    amax = np.abs(v).max(axis=1)
    e = np.array([row_exponent(float(a)) for a in amax])
    with pytest.raises(ValueError):
        e4m3_encode(v * np.exp2(-(e - 1).astype(np.float64))[:, None])
    assert np.all(amax * np.exp2(-(e + 1).astype(np.float64)) <= 224)
    fine = _from_bits(roundtrip_rows(_bf16_bits(v)))
    rel = np.abs(fine - v).max() / np.abs(v).max()
    assert 0 < rel <= 2.0 ** -4
