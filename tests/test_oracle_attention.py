"""Pins of the oracle's fp64 attention: closed forms, permutation invariance,
a library routine (scaled_dot_product_attention in fp64 on the CPU) and a
brute-force loop on tiny inputs; plus the end-to-end check that the paged
concatenation equals a flat, page-free concatenation."""

import math
import random

import numpy as np
import pytest
import torch

from oracle import PagedCacheOracle, StreamConfig, attend_fp64, gather_visible
from oracle.attention import softmax_rows_fp64
from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS, frame_tensor, is_keyframe
from synth.inputs import bf16_bits_to_f64
from tests.bruteforce import FlatFrameModel


def bf16(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def rand_bits(rng, *shape, scale=1.0):
    return bf16(rng.standard_normal(shape) * scale)


def sdpa_fp64(q_bits, k_bits, v_bits, sm_scale):
    q = torch.from_numpy(bf16_bits_to_f64(q_bits)).permute(1, 0, 2)
    k = torch.from_numpy(bf16_bits_to_f64(k_bits)).permute(1, 0, 2)
    v = torch.from_numpy(bf16_bits_to_f64(v_bits)).permute(1, 0, 2)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=sm_scale)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("seed", range(5))
def test_matches_library_sdpa(seed):
    rng = np.random.default_rng(seed)
    n_q, n, h, d = 37, 301, 3, 64
    q, k, v = rand_bits(rng, n_q, h, d), rand_bits(rng, n, h, d), rand_bits(rng, n, h, d)
    for scale in (0.125, 0.7, 2.0):
        np.testing.assert_allclose(attend_fp64(q, k, v, scale), sdpa_fp64(q, k, v, scale),
                                   rtol=0, atol=1e-12)


def test_brute_force_loop():
    rng = np.random.default_rng(3)
    q, k, v = rand_bits(rng, 2, 1, 4), rand_bits(rng, 3, 1, 4), rand_bits(rng, 3, 1, 4)
    Q, K, V = bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v)
    out = attend_fp64(q, k, v, 0.5)
    for i in range(2):
        w = [math.exp(0.5 * sum(Q[i, 0, c] * K[j, 0, c] for c in range(4))) for j in range(3)]
        for c in range(4):
            ref = sum(w[j] * V[j, 0, c] for j in range(3)) / sum(w)
            assert abs(out[i, 0, c] - ref) < 1e-13


def test_rows_sum_to_one():
    rng = np.random.default_rng(1)
    q, k = rand_bits(rng, 50, 2, 64), rand_bits(rng, 400, 2, 64)
    for h in range(2):
        p = softmax_rows_fp64(q, k, 0.125, h)
        assert np.abs(p.sum(axis=1) - 1).max() < 1e-12
        assert (p >= 0).all()


def test_closed_forms():
    rng = np.random.default_rng(2)
    k, v = rand_bits(rng, 97, 2, 64), rand_bits(rng, 97, 2, 64)
    V = bf16_bits_to_f64(v)
    # q = 0: uniform weights, the mean of the visible values
    zero_q = np.zeros((5, 2, 64), np.uint16)
    np.testing.assert_allclose(attend_fp64(zero_q, k, v, 0.125), np.broadcast_to(V.mean(0), (5, 2, 64)),
                               atol=1e-14)
    # a single visible token: its value
    q = rand_bits(rng, 5, 2, 64)
    np.testing.assert_allclose(attend_fp64(q, k[:1], v[:1], 0.125), np.broadcast_to(V[0], (5, 2, 64)),
                               atol=0)
    # every key identical: the mean of the values
    same_k = np.broadcast_to(k[:1], k.shape).copy()
    np.testing.assert_allclose(attend_fp64(q, same_k, v, 0.125), np.broadcast_to(V.mean(0), (5, 2, 64)),
                               atol=1e-14)
    # scores far apart: the max-subtraction keeps exp finite; one key dominates
    big_q = bf16(np.full((1, 1, 64), 8.0))
    big_k = bf16(np.concatenate([np.full((1, 1, 64), 8.0), np.full((3, 1, 64), -8.0)]))
    vv = rand_bits(rng, 4, 1, 64)
    out = attend_fp64(big_q, big_k, vv, 1.0)
    np.testing.assert_allclose(out[0, 0], bf16_bits_to_f64(vv)[0, 0], atol=0)


def test_page_permutation_invariance():
    """Any reordering of the visible pages gives the same result (up to fp64 rounding)."""
    rng = np.random.default_rng(4)
    ps, n_pages = 16, 9
    q = rand_bits(rng, 22, 4, 64)
    k, v = rand_bits(rng, n_pages * ps, 4, 64), rand_bits(rng, n_pages * ps, 4, 64)
    base = attend_fp64(q, k, v, 0.125)
    for trial in range(5):
        perm = np.random.default_rng(trial).permutation(n_pages)
        rows = (perm[:, None] * ps + np.arange(ps)[None, :]).reshape(-1)
        np.testing.assert_allclose(attend_fp64(q, k[rows], v[rows], 0.125), base, atol=1e-12)


def test_sampled_rows_match_full():
    rng = np.random.default_rng(5)
    q, k, v = rand_bits(rng, 40, 2, 64), rand_bits(rng, 90, 2, 64), rand_bits(rng, 90, 2, 64)
    full = attend_fp64(q, k, v, 0.125)
    rows = [0, 7, 39]
    np.testing.assert_array_equal(attend_fp64(q, k, v, 0.125, rows=rows), full[rows])


@pytest.mark.parametrize("seed", range(6))
def test_paged_concat_equals_flat_concat(seed):
    """The oracle's paged gather, through appends, rollbacks and evictions, gives
    the same attention as the page-free flat model's token list."""
    w = WORKLOADS["tiny"]
    rng = random.Random(seed)
    kf = rng.randint(1, 3)
    o = PagedCacheOracle(w.pool_pages, w.page_size)
    cfg = StreamConfig(mode="frame", num_scale=w.num_scale, window=w.window, n_patch=w.n_patch,
                       n_special=w.n_special)
    sid = o.open_stream(cfg)
    flat = FlatFrameModel(w.num_scale, w.window, w.n_patch, w.n_special)
    gen = {}

    def lookup(s, f, layer):
        if (s, f) not in gen:
            gen[(s, f)] = (frame_tensor(seed, 0, s, layer, f, TENSOR_K, w.frame_tokens, w.heads, 64),
                           frame_tensor(seed, 0, s, layer, f, TENSOR_V, w.frame_tokens, w.heads, 64))
        return gen[(s, f)]

    for t in range(w.frames):
        o.append_frame(sid, t, w.frame_tokens)
        flat.append(sid, t)
        q = frame_tensor(seed, 0, sid, 0, t, TENSOR_Q, w.frame_tokens, w.heads, 64)
        kp, vp = gather_visible(o.visible_tokens(sid), 0, lookup)
        kf_, vf_ = gather_visible(sorted(flat.visible().elements()), 0, lookup)
        np.testing.assert_allclose(attend_fp64(q, kp, vp, w.sm_scale),
                                   attend_fp64(q, kf_, vf_, w.sm_scale), atol=1e-12)
        if is_keyframe(t, w.num_scale, kf):
            o.evict_window(sid); flat.evict()
        else:
            o.rollback_last_frame(sid); flat.rollback()
