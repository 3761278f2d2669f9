"""Pins of the seeded input generator (shared by the oracle and the CUDA
library's own generator): splitmix64 against its published sequence, exact
bf16 rounding against torch's conversion, and the Irwin-Hall moments."""

import numpy as np
import pytest
import torch

from synth import WORKLOADS, frame_tensor, multistream_schedule, pack_key, splitmix64
from synth.inputs import _f32_to_bf16_bits, bf16_bits_to_f32, gaussian_bf16


def test_splitmix64_published_sequence():
    # The reference sequence of splitmix64 seeded with 1234567 (state advanced by
    # the golden gamma before each output).
    expected = [6457827717110365317, 3203168211198807973, 9817491932198370423,
                4593380528125082431, 16408922859458223821]
    gamma = 0x9E3779B97F4A7C15
    states = np.array([(1234567 + i * gamma) % (1 << 64) for i in range(5)], dtype=np.uint64)
    assert [int(x) for x in splitmix64(states)] == expected


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 3,
                        # exact ties between two bf16 values: round to even
                        (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)])
    ours = _f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_gaussian_moments_and_range():
    keys = pack_key(0, 1, 0, 0, 0, 1, np.arange(2000)[:, None], np.arange(25)[None, :] % 32, 0)
    x = bf16_bits_to_f32(gaussian_bf16(keys.reshape(-1))).astype(np.float64)
    assert abs(x.mean()) < 0.03
    assert abs(x.var() - 1.0) < 0.03
    assert np.abs(x).max() <= 2 * 1.7320508 + 1e-6     # Irwin-Hall support: 4 uniforms


def test_query_scale_is_exact():
    a = frame_tensor(0, 1, 0, 0, 5, 0, 10, 4, 64)
    b = frame_tensor(0, 1, 0, 0, 5, 0, 10, 4, 64, scale=0.125)
    np.testing.assert_array_equal(bf16_bits_to_f32(a) * np.float32(0.125), bf16_bits_to_f32(b))


def test_key_fields_are_distinct_and_checked():
    k1 = pack_key(1, 2, 3, 4, 5, 1, 6, 7, 8)
    k2 = pack_key(1, 2, 3, 4, 5, 2, 6, 7, 8)
    assert int(k1) != int(k2)
    assert int(pack_key(127, 7, 63, 31, 65535, 3, 16383, 31, 63)) == (1 << 64) - 1
    with pytest.raises(ValueError):
        pack_key(0, 0, 0, 0, 65536, 0, 0, 0, 0)
    with pytest.raises(ValueError):
        pack_key(0, 0, 0, 0, 0, 0, 0, 0, 64)


def test_multistream_schedule():
    sched = multistream_schedule(0)
    assert len(sched) == WORKLOADS["multistream"].streams
    assert all(100 <= n <= 5000 and kf in (1, 2, 4, 8) for n, kf in sched)
    assert sched == multistream_schedule(0) and sched != multistream_schedule(1)
