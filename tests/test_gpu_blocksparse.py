"""pkv_attend_blocksparse: attention over the scale pages and the `keep` pages with
the highest estimated attention mass (vLLM-Omni RFC "Reconstruction Engine",
section 5: Sparse-VGGT block skipping, FastVGGT anchors). The kept table
positions must equal the oracle's bit for bit (oracle/blocksparse.py computes the
same fp32 estimate in the same order), and the output must match the fp64 oracle
over the kept pages; keep >= the visible pages is pkv_attend exactly."""

import random

import numpy as np
import pytest
import torch

from oracle import attend_fp64, gather_visible
from oracle.blocksparse import kept_positions, page_scores, visible_tokens_blocksparse
from synth import WORKLOADS, is_keyframe
from tests.pairing import Pair, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_build_gb300 import build
    build.build()


def _stream(pr, frames):
    sid = pr.open()
    for t in range(frames):
        pr.append(sid, t)
        if t < frames - 1:
            pr.evict(sid)
    return sid


def _check(pr, sid, layer, t, keep, rows=None):
    q = pr.gpu_q_chunk(sid, layer, [t])
    qb = pr.cpu_q(sid, layer, [t])
    out = pr.gpu.attend_blocksparse(q, sid, layer, keep=keep, sm_scale=pr.w.sm_scale)
    got = pr.gpu.blocksparse_kept()
    n_anchor = len(pr.ora._stream(sid, "frame").scale)
    ref = kept_positions(page_scores(pr.ora, sid, layer, qb, pr.lookup), n_anchor, keep)
    assert got == ref, f"kept positions differ (keep {keep})"
    toks = visible_tokens_blocksparse(pr.ora, sid, layer, qb, keep, pr.lookup)
    k, v = gather_visible(toks, layer, pr.lookup)
    o = attend_fp64(qb, k, v, pr.w.sm_scale, rows=rows)
    e = attend_fp64(qb, k, v & np.uint16(0x7FFF), pr.w.sm_scale, rows=rows)
    sel = out if rows is None else out[torch.from_numpy(rows).cuda()]
    assert_close(sel, o, e, f"layer {layer} keep {keep}")
    return out


def test_tiny_against_oracle():
    w = WORKLOADS["tiny"]
    pr = Pair(w, seed=7, layers=2)
    sid = _stream(pr, 11)
    for layer in (0, 1):
        for keep in (0, 1, 2, 3, 100):
            _check(pr, sid, layer, 10, keep)
    pr.gpu.sync()


def test_lingbot_against_oracle():
    w = WORKLOADS["lingbot"]
    pr = Pair(w, seed=8, layers=2, pool_pages=256)
    sid = _stream(pr, 120)
    rows = np.arange(0, w.frame_tokens, 7)
    for layer in (0, 1):
        for keep in (4, 16, 40):
            _check(pr, sid, layer, 119, keep, rows=rows)
    pr.gpu.sync()


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_mean_key_cache_follows_every_page_change(seed):
    """Estimates on both layers at every frame of a stream with rollbacks,
    evictions and windowed resets (which copy rows into freshly popped pages): a
    call reuses the mean keys an earlier call cached for the pages that did not
    change, and its kept list must still equal the oracle's, which recomputes
    every page. A rolled-back frame's patch page goes back to the free stack and
    is popped again by the next frame at the same length, so a page whose rows
    changed without its cached value being dropped would show up here."""
    rng = random.Random(seed)
    S = rng.randint(1, 2)
    w = WORKLOADS["tiny"].with_(page_size=32, n_patch=32, n_special=rng.choice([2, 4, 6]), num_scale=S,
                                window=rng.randint(2, 4), heads=rng.choice([2, 4]),
                                window_slots=rng.randint(S + 2, 7), overlap_keyframes=rng.randint(0, S))
    pr = Pair(w, seed, layers=2, pool_pages=96)
    sid = pr.open()
    kf = rng.randint(1, 3)
    for t in range(36):
        pr.append(sid, t)
        n_pages = pr.gpu.visible_count(sid)[0]
        for layer in (0, 1):
            keep = rng.randint(0, n_pages)
            if t % 6 == 5:
                _check(pr, sid, layer, t, keep)
            else:
                # kept lists only (the attention of the kept pages is checked above)
                q = pr.gpu_q_chunk(sid, layer, [t])
                pr.gpu.attend_blocksparse(q, sid, layer, keep=keep, sm_scale=w.sm_scale)
                n_anchor = len(pr.ora._stream(sid, "frame").scale)
                ref = kept_positions(page_scores(pr.ora, sid, layer, pr.cpu_q(sid, layer, [t]), pr.lookup),
                                     n_anchor, keep)
                assert pr.gpu.blocksparse_kept() == ref, f"seed {seed} frame {t} layer {layer}"
        if is_keyframe(t, S, kf) and rng.random() > 0.2:
            pr.evict(sid)
        else:
            pr.rollback(sid)
    pr.gpu.sync()


def test_keep_everything_is_pkv_attend():
    w = WORKLOADS["lingbot"]
    pr = Pair(w, seed=9, pool_pages=256)
    sid = _stream(pr, 90)
    q = pr.gpu_q_chunk(sid, 0, [89])
    full = pr.gpu.attend(q, sid, 0, sm_scale=w.sm_scale)
    sparse = pr.gpu.attend_blocksparse(q, sid, 0, keep=1000, sm_scale=w.sm_scale)
    assert torch.equal(full, sparse)
    n = pr.gpu.visible_count(sid)[0]
    assert pr.gpu.blocksparse_kept() == list(range(n))
    pr.gpu.sync()


def test_errors():
    from paged_kv_cache_build_gb300 import PkvError, chunked_stream_cfg
    w = WORKLOADS["tiny"]
    pr = Pair(w, layers=1)
    with pytest.raises(PkvError) as ei:
        pr.gpu.blocksparse_kept()                                          # no call yet
    assert ei.value.code == "STATE"
    sid = _stream(pr, 3)
    q = pr.gpu_q_chunk(sid, 0, [2])
    with pytest.raises(PkvError) as ei:
        pr.gpu.attend_blocksparse(q, sid, 0, keep=-1)
    assert ei.value.code == "INVALID"
    cid = pr.gpu.open_stream(chunked_stream_cfg(2, 2, w.frame_tokens))
    with pytest.raises(PkvError) as ei:
        pr.gpu.attend_blocksparse(q, cid, 0, keep=1)
    assert ei.value.code == "STATE"
    pr.gpu.sync()
