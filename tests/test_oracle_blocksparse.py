"""Pins of the oracle's page skipping by estimated attention mass (vLLM-Omni RFC
"Reconstruction Engine", section 5: Sparse-VGGT block skipping, FastVGGT anchors):
the fp32 estimate's defined order, the ranking rule against brute force, the
keep-all and keep-none limits, and a planted page that the estimate must find."""

import math

import numpy as np
import pytest
import torch

from oracle import PagedCacheOracle, StreamConfig
from oracle.blocksparse import (kept_positions, page_score, page_scores, pooled_mean,
                                visible_tokens_blocksparse)


def bf16(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_pooled_mean_exact_and_close():
    rows = bf16([[[1.0, -2.0]], [[2.0, 4.0]], [[3.0, 7.0]]])      # [3][1][2]
    np.testing.assert_array_equal(pooled_mean(rows), np.array([[2.0, 3.0]], dtype=np.float32))
    rng = np.random.default_rng(0)
    r = bf16(rng.standard_normal((250, 4, 64)))
    ref = r.astype(np.uint32) << 16
    ref = ref.view(np.float32).astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(pooled_mean(r), ref, rtol=0, atol=1e-5)


def test_score_order_is_sequential_fp32():
    """1e8 + 1 - 1e8 in one running fp32 total is 0 (the 1 is absorbed): the
    estimate is the sequential sum, not the exact one."""
    qm = np.array([[1e8, 1.0, -1e8]], dtype=np.float32)
    km = np.ones((1, 3), dtype=np.float32)
    assert page_score(qm, km) == np.float32(0.0)
    assert page_score(np.ones((2, 64), np.float32), np.ones((2, 64), np.float32)) == 128.0
    # products are rounded before the add: 3 * (1 + 2^-12)^2 rounds to fp32 first
    a = np.float32(1 + 2.0 ** -12)
    assert page_score(np.array([[a]], np.float32), np.array([[a]], np.float32)) == np.float32(a * a)


def test_score_sums_each_head_first():
    """The heads' sums are formed first, then added in head order: with head 0's
    products (1e8, 0) and head 1's (-1e8, 1), head 1's sum is -1e8 (the 1 is
    absorbed: fp32 spacing at 1e8 is 8), so the score is 1e8 + (-1e8) = 0; one
    running sum over all products in order would give 1e8 + 0 - 1e8 + 1 = 1."""
    qm = np.array([[1e8, 0.0], [-1e8, 1.0]], dtype=np.float32)
    km = np.ones((2, 2), dtype=np.float32)
    assert page_score(qm, km) == np.float32(0.0)


def test_ranking_rule_brute_force():
    rng = np.random.default_rng(1)
    for trial in range(200):
        n = int(rng.integers(1, 40))
        anchors = int(rng.integers(0, min(n, 8) + 1))
        s = rng.integers(-5, 6, size=n).astype(np.float32)        # many ties
        if trial % 7 == 0 and n > anchors:
            s[rng.integers(anchors, n)] = np.nan
        keep = int(rng.integers(0, n + 3))
        got = kept_positions(list(s), anchors, keep)
        # brute force: e is kept if fewer than `keep` candidates beat it
        def beats(o, e):
            ko = -math.inf if math.isnan(s[o]) else s[o]
            ke = -math.inf if math.isnan(s[e]) else s[e]
            return ko > ke or (ko == ke and o < e)
        ref = [e for e in range(n) if e < anchors or
               sum(beats(o, e) for o in range(anchors, n) if o != e) < keep]
        assert got == ref
        assert len(got) == anchors + min(max(keep, 0), n - anchors)


def _tiny_stream(frames, planted=None):
    """Tiny frame-mode stream of the cache oracle with Gaussian K/V; the keys of
    frame `planted` (if any) point along the query direction."""
    H, D, n_patch, n_sp = 2, 64, 16, 6
    rng = np.random.default_rng(5)
    u = rng.standard_normal((H, D))
    kv = {}
    for f in range(frames):
        k = rng.standard_normal((n_patch + n_sp, H, D))
        if f == planted:
            k = 0.2 * k + 3.0 * u[None]
        kv[f] = (bf16(k), bf16(rng.standard_normal((n_patch + n_sp, H, D))))
    q = bf16(u[None] + 0.5 * rng.standard_normal((n_patch + n_sp, H, D)))
    ora = PagedCacheOracle(64, 16)
    sid = ora.open_stream(StreamConfig(mode="frame", num_scale=2, window=4, n_patch=n_patch,
                                       n_special=n_sp))
    for f in range(frames):
        ora.append_frame(sid, f, n_patch + n_sp)
        if f < frames - 1:
            ora.evict_window(sid)
    return ora, sid, q, (lambda s, f, layer: kv[f])


def test_planted_page_is_found():
    """Window page of the planted frame (keys along the queries): the highest
    estimate, so keep = 1 keeps the anchors and exactly that page."""
    ora, sid, q, lookup = _tiny_stream(8, planted=5)
    idx, lens = ora.visible_table(sid)
    scores = page_scores(ora, sid, 0, q, lookup)
    planted_e = [e for e, p in enumerate(idx) if ora.slots[p][0] == (sid, 5, 0)]
    assert len(planted_e) == 1
    cand = list(range(2, len(idx)))
    assert max(cand, key=lambda e: scores[e]) == planted_e[0]
    assert kept_positions(scores, 2, 1) == [0, 1, planted_e[0]]


def test_keep_all_and_keep_none():
    ora, sid, q, lookup = _tiny_stream(9)
    n = len(ora.visible_table(sid)[0])
    assert visible_tokens_blocksparse(ora, sid, 0, q, n, lookup) == ora.visible_tokens(sid)
    anchors_only = visible_tokens_blocksparse(ora, sid, 0, q, 0, lookup)
    assert anchors_only == [t for t in ora.visible_tokens(sid) if t[1] < 2 and t[2] < 16]
