"""Pins of the oracle's intra-frame attention (vLLM-Omni RFC "Reconstruction
Engine", sections 2.2 and 3.3: each frame's tokens attend to their own frame
only). Checked against a library routine given the block-diagonal mask over all
frames at once, closed forms, a brute-force loop, permutations, and the paged
cache oracle's first frame, whose visible tokens are exactly its own."""

import math

import numpy as np
import pytest
import torch

from oracle import PagedCacheOracle, StreamConfig, attend_fp64, frame_attend_fp64, gather_visible
from synth import TENSOR_K, TENSOR_Q, TENSOR_V, frame_tensor
from synth.inputs import bf16_bits_to_f64


def bf16(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def rand_bits(rng, *shape, scale=1.0):
    return bf16(rng.standard_normal(shape) * scale)


@pytest.mark.parametrize("seed", range(3))
def test_block_diagonal_sdpa(seed):
    """All frames' tokens in one sequence, attention restricted by a
    block-diagonal mask (torch's fp64 scaled_dot_product_attention)."""
    rng = np.random.default_rng(seed)
    F, T, H, D = 3, 29, 2, 64
    q, k, v = (rand_bits(rng, F, T, H, D) for _ in range(3))
    got = frame_attend_fp64(q, k, v, 0.3)
    Q, K, V = (torch.from_numpy(bf16_bits_to_f64(x).reshape(F * T, H, D)).permute(1, 0, 2)
               for x in (q, k, v))
    frame_of = torch.arange(F * T) // T
    mask = frame_of[:, None] == frame_of[None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=0.3)
    ref = ref.permute(1, 0, 2).reshape(F, T, H, D).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_brute_force_loop():
    rng = np.random.default_rng(7)
    q, k, v = rand_bits(rng, 2, 3, 1, 4), rand_bits(rng, 2, 3, 1, 4), rand_bits(rng, 2, 3, 1, 4)
    Q, K, V = bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v)
    out = frame_attend_fp64(q, k, v, 0.5)
    for f in range(2):
        for i in range(3):
            w = [math.exp(0.5 * sum(Q[f, i, 0, c] * K[f, j, 0, c] for c in range(4))) for j in range(3)]
            for c in range(4):
                ref = sum(w[j] * V[f, j, 0, c] for j in range(3)) / sum(w)
                assert abs(out[f, i, 0, c] - ref) < 1e-13


def test_one_token_frames_return_their_value():
    """A frame of one token: the softmax over one key is 1, so out = v."""
    rng = np.random.default_rng(1)
    q, k, v = (rand_bits(rng, 5, 1, 3, 64) for _ in range(3))
    np.testing.assert_array_equal(frame_attend_fp64(q, k, v, 0.125), bf16_bits_to_f64(v))


def test_equal_keys_give_the_mean_value():
    """Identical keys within a frame: uniform weights, out = mean of the frame's v."""
    rng = np.random.default_rng(2)
    F, T, H, D = 2, 17, 2, 64
    q, v = rand_bits(rng, F, T, H, D), rand_bits(rng, F, T, H, D)
    k = np.repeat(rand_bits(rng, F, 1, H, D), T, axis=1)
    got = frame_attend_fp64(q, k, v, 0.7)
    mean = bf16_bits_to_f64(v).mean(axis=1, keepdims=True)
    np.testing.assert_allclose(got, np.broadcast_to(mean, got.shape), rtol=0, atol=1e-13)


def test_frames_do_not_see_each_other():
    """Changing one frame's keys and values leaves every other frame's output
    unchanged, and permuting frames (or a frame's tokens) permutes the output."""
    rng = np.random.default_rng(3)
    F, T, H, D = 4, 11, 2, 64
    q, k, v = (rand_bits(rng, F, T, H, D) for _ in range(3))
    base = frame_attend_fp64(q, k, v, 0.25)
    k2, v2 = k.copy(), v.copy()
    k2[2], v2[2] = rand_bits(rng, T, H, D), rand_bits(rng, T, H, D)
    moved = frame_attend_fp64(q, k2, v2, 0.25)
    for f in (0, 1, 3):
        np.testing.assert_array_equal(moved[f], base[f])
    assert np.abs(moved[2] - base[2]).max() > 1e-3
    perm = np.array([2, 0, 3, 1])
    np.testing.assert_allclose(frame_attend_fp64(q[perm], k[perm], v[perm], 0.25), base[perm],
                               rtol=0, atol=1e-13)
    tp = rng.permutation(T)
    np.testing.assert_allclose(frame_attend_fp64(q[:, tp], k[:, tp], v[:, tp], 0.25), base[:, tp],
                               rtol=0, atol=1e-13)


def test_first_frame_of_a_stream_is_frame_attention():
    """The cache oracle's first frame sees only its own tokens (scale page plus
    its special tokens), so its global attention is the frame attention."""
    H, D, n_patch, n_sp = 4, 64, 16, 6
    ora = PagedCacheOracle(32, 16)
    sid = ora.open_stream(StreamConfig(mode="frame", num_scale=2, window=4, n_patch=n_patch,
                                       n_special=n_sp))
    T = n_patch + n_sp
    ora.append_frame(sid, 0, T)
    toks = ora.visible_tokens(sid)
    assert sorted(t for (_, _, t) in toks) == list(range(T))
    kv = {f: (frame_tensor(9, 0, sid, 0, f, TENSOR_K, T, H, D), frame_tensor(9, 0, sid, 0, f, TENSOR_V, T, H, D))
          for f in (0,)}
    K, V = gather_visible(toks, 0, lambda s, f, layer: kv[f])
    q = frame_tensor(9, 0, sid, 0, 0, TENSOR_Q, T, H, D, 0.125)
    paged = attend_fp64(q, K, V, 0.125)
    framed = frame_attend_fp64(q[None], kv[0][0][None], kv[0][1][None], 0.125)[0]
    np.testing.assert_allclose(paged, framed, rtol=0, atol=1e-13)


def test_shape_errors():
    z = np.zeros((2, 3, 1, 64), dtype=np.uint16)
    with pytest.raises(ValueError):
        frame_attend_fp64(z, z[:1], z, 1.0)
    with pytest.raises(ValueError):
        frame_attend_fp64(z[0], z[0], z[0], 1.0)
