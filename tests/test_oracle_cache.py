"""Pins of the oracle's page state machine against things other than itself:
a hand-derived trace, a brute-force flat model without pages, and invariants
the article fixes (page-type counts, table order, constant patch cache,
append + rollback identity, all-or-nothing errors)."""

import math
import os
import random
from collections import Counter

import pytest

from oracle import OracleError, PagedCacheOracle, StreamConfig
from synth import WORKLOADS, is_keyframe
from tests.bruteforce import FlatChunkModel, FlatFrameModel

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def frame_cfg(w, **kw):
    base = dict(mode="frame", num_scale=w.num_scale, window=w.window, n_patch=w.n_patch,
                n_special=w.n_special, window_slots=w.window_slots,
                overlap_keyframes=w.overlap_keyframes)
    base.update(kw)
    return StreamConfig(**base)


def check_pool(o):
    """Every page is either free or held by exactly one stream, once."""
    held = []
    for sid in o.streams:
        idx, _ = o.visible_table(sid)
        held += idx
    assert len(set(o.free)) == len(o.free)
    assert len(set(held)) == len(held)
    assert set(o.free).isdisjoint(held)
    assert len(o.free) + len(held) == o.P


def test_tiny_golden_trace():
    w = WORKLOADS["tiny"]
    rows = []
    with open(os.path.join(GOLDEN, "tiny_trace.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            cols = [c.strip() for c in line.split("|")]
            rows.append([[] if c == "-" else [int(x) for x in c.split()] for c in cols])
    assert len(rows) == w.frames
    o = PagedCacheOracle(w.pool_pages, w.page_size)
    sid = o.open_stream(frame_cfg(w))
    for t, (fr, scale, window, special, sp_lens, freed) in enumerate(rows):
        assert fr == [t]
        o.append_frame(sid, t, w.frame_tokens)
        idx, lens = o.visible_table(sid)
        assert idx == scale + window + special
        assert lens == [w.page_size] * (len(scale) + len(window)) + sp_lens
        before = set(o.free)
        o.evict_window(sid)
        assert sorted(set(o.free) - before) == freed
        check_pool(o)
    assert sum(lens) == 168


def _random_frame_run(rng, o, sid, model, cfg, n_frames, kf, rollback_prob=0.0):
    for t in range(n_frames):
        o.append_frame(sid, t, cfg.n_patch + cfg.n_special)
        model.append(sid, t)
        assert Counter(o.visible_tokens(sid)) == model.visible()
        check_pool(o)
        keep = is_keyframe(t, cfg.num_scale, kf) and rng.random() >= rollback_prob
        if keep:
            o.evict_window(sid)
            model.evict()
        else:
            o.rollback_last_frame(sid)
            model.rollback()
        assert Counter(o.visible_tokens(sid)) == model.visible()
        check_pool(o)


@pytest.mark.parametrize("seed", range(40))
def test_frame_mode_matches_flat_model(seed):
    rng = random.Random(seed)
    ps = rng.choice([8, 16])
    cfg = StreamConfig(mode="frame", num_scale=rng.randint(1, 3), window=rng.randint(1, 5),
                       n_patch=ps, n_special=rng.randint(1, 6))
    o = PagedCacheOracle(64, ps)
    sid = o.open_stream(cfg)
    model = FlatFrameModel(cfg.num_scale, cfg.window, cfg.n_patch, cfg.n_special)
    _random_frame_run(rng, o, sid, model, cfg, rng.randint(1, 40), rng.randint(1, 4), 0.2)


@pytest.mark.parametrize("seed", range(20))
def test_windowed_mode_matches_flat_model(seed):
    rng = random.Random(1000 + seed)
    ps = rng.choice([8, 16])
    S = rng.randint(1, 4)
    cfg = StreamConfig(mode="frame", num_scale=S, window=rng.randint(1, 6), n_patch=ps,
                       n_special=rng.randint(1, 6), window_slots=rng.randint(S + 1, 12),
                       overlap_keyframes=rng.randint(0, S))
    o = PagedCacheOracle(96, ps)
    sid = o.open_stream(cfg)
    model = FlatFrameModel(cfg.num_scale, cfg.window, cfg.n_patch, cfg.n_special,
                           cfg.window_slots, cfg.overlap_keyframes)
    _random_frame_run(rng, o, sid, model, cfg, rng.randint(10, 60), rng.randint(1, 3), 0.1)
    st = o.streams[sid]
    assert st.kept < cfg.window_slots


@pytest.mark.parametrize("seed", range(20))
def test_chunked_mode_matches_flat_model(seed):
    rng = random.Random(2000 + seed)
    ps = rng.choice([8, 16])
    cfg = StreamConfig(mode="chunked", chunk_size=rng.randint(1, 4),
                       sliding_window_num=rng.randint(1, 4), tokens_per_frame=rng.randint(1, 20))
    o = PagedCacheOracle(128, ps)
    sid = o.open_stream(cfg)
    model = FlatChunkModel(cfg.sliding_window_num, cfg.tokens_per_frame)
    fid = 0
    for _ in range(rng.randint(1, 12)):
        for _f in range(cfg.chunk_size):
            o.append_frame(sid, fid, cfg.tokens_per_frame)
            model.append(sid, fid)
            if rng.random() < 0.2:
                o.rollback_last_frame(sid)
                model.rollback()
            else:
                fid += 1
            assert Counter(o.visible_tokens(sid)) == model.visible()
            check_pool(o)
        # pages are packed: each chunk uses exactly ceil(tokens / page_size) pages
        for c in o.streams[sid].chunks:
            assert len(c.pages) == math.ceil(c.length / ps)
        o.evict_window(sid)
        model.evict()
        assert Counter(o.visible_tokens(sid)) == model.visible()
        assert len(o.streams[sid].chunks) <= cfg.sliding_window_num - 1
        check_pool(o)


def test_lingbot_page_counts_and_order():
    """Section 2: 8 scale pages, a 64-page window, special pages holding exactly
    42 frames x 6 tokens, a patch cache that stops growing, table order."""
    w = WORKLOADS["lingbot"]
    o = PagedCacheOracle(w.pool_pages, w.page_size)
    sid = o.open_stream(frame_cfg(w))
    f_sp = w.page_size // w.n_special
    assert f_sp == 42 and f_sp * w.n_special == 252
    for t in range(w.frames):
        o.append_frame(sid, t, w.frame_tokens)
        st = o.streams[sid]
        idx, lens = o.visible_table(sid)
        n_patch = len(st.scale) + len(st.window)
        assert len(st.scale) == min(t + 1, 8)
        assert len(st.window) <= 64
        if t >= w.num_scale + w.window - 1:
            assert n_patch == w.num_scale + w.window        # 72 while attending
        assert len(st.special) == math.ceil((t + 1) / 42)
        assert all(n == 252 for n in lens[n_patch:-1])
        assert lens[-1] == 6 * ((t % 42) + 1)
        # order: scale pages, then the window oldest first, then special pages
        toks = o.visible_tokens(sid)
        frames_in_order = [f for (_, f, tk) in toks if tk < w.n_patch][::w.n_patch]
        assert frames_in_order == list(range(min(t + 1, 8))) + list(range(max(8, t - 63), t + 1))
        sp_frames = [f for (_, f, tk) in toks if tk >= w.n_patch][::w.n_special]
        assert sp_frames == list(range(t + 1))
        o.evict_window(sid)
        if t >= w.num_scale + w.window - 1:
            assert o.patch_pages_in_use(sid) == w.num_scale + w.window - 1   # 71 between frames
        check_pool(o)
    # visible tokens at the last frame: 8*256 + 64*256 + 512*6
    assert sum(lens) == 21504


@pytest.mark.parametrize("length", [100, 400, 1000, 3000])
def test_patch_cache_constant_with_length(length):
    """Section 2 (and the memory sweep of section 5): the patch cache does not
    grow with stream length; only the append-only special pages do, by
    ceil(kept / 42)."""
    w = WORKLOADS["lingbot"]
    o = PagedCacheOracle(1024, w.page_size)
    sid = o.open_stream(frame_cfg(w))
    for t in range(length):
        o.append_frame(sid, t, w.frame_tokens)
        o.evict_window(sid)
    assert o.patch_pages_in_use(sid) == 71
    assert len(o.streams[sid].special) == math.ceil(length / 42)


def test_keyframes_cut_cache_growth():
    """Section 3: with keyframe interval N the special stream grows ~1/N as fast,
    and non-keyframes leave no trace."""
    w = WORKLOADS["long"].with_(frames=2000)
    o = PagedCacheOracle(512, w.page_size)
    sid = o.open_stream(frame_cfg(w))
    kept = 0
    for t in range(w.frames):
        o.append_frame(sid, t, w.frame_tokens)
        if is_keyframe(t, w.num_scale, w.keyframe_interval):
            o.evict_window(sid)
            kept += 1
        else:
            o.rollback_last_frame(sid)
    assert kept == 8 + math.ceil((2000 - 8) / 4)
    assert len(o.streams[sid].special) == math.ceil(kept / 42)
    assert o.patch_pages_in_use(sid) == 71


def test_append_rollback_identity():
    """Section 3: append -> (attend) -> rollback leaves metadata and every valid
    slot exactly as before, including across a new special page."""
    w = WORKLOADS["tiny"]
    o = PagedCacheOracle(w.pool_pages, w.page_size)
    sid = o.open_stream(frame_cfg(w))
    for t in range(w.frames):
        before = o.snapshot()
        o.append_frame(sid, 100 + t, w.frame_tokens)
        o.rollback_last_frame(sid)
        assert o.snapshot() == before
        o.append_frame(sid, t, w.frame_tokens)
        o.evict_window(sid)
    with pytest.raises(OracleError) as e:
        o.rollback_last_frame(sid)        # eviction committed the frame
    assert e.value.code == "STATE"


def test_errors_leave_state_unchanged():
    w = WORKLOADS["tiny"]
    o = PagedCacheOracle(5, w.page_size)
    sid = o.open_stream(frame_cfg(w))
    with pytest.raises(OracleError) as e:
        o.append_frame(sid, 0, 21)
    assert e.value.code == "INVALID"
    o.append_frame(sid, 0, 22); o.evict_window(sid)      # pops 2 pages
    o.append_frame(sid, 1, 22); o.evict_window(sid)      # pops 1
    o.append_frame(sid, 2, 22); o.evict_window(sid)      # pops 2 -> 0 free
    snap = o.snapshot()
    with pytest.raises(OracleError) as e:
        o.append_frame(sid, 3, 22)
    assert e.value.code == "OOM"
    assert o.snapshot() == snap
    # window full without an eviction
    o2 = PagedCacheOracle(64, 16)
    s2 = o2.open_stream(StreamConfig(mode="frame", num_scale=0, window=2, n_patch=16, n_special=6))
    o2.append_frame(s2, 0, 22)
    o2.append_frame(s2, 1, 22)
    snap = o2.snapshot()
    with pytest.raises(OracleError) as e:
        o2.append_frame(s2, 2, 22)
    assert e.value.code == "STATE"
    assert o2.snapshot() == snap


def test_multistream_batch_equals_sequential():
    """A batched multi-stream append is the sequence of single appends in the
    order given, validated as a whole."""
    w = WORKLOADS["tiny"]
    a = PagedCacheOracle(200, w.page_size)
    b = PagedCacheOracle(200, w.page_size)
    sa = [a.open_stream(frame_cfg(w)) for _ in range(5)]
    sb = [b.open_stream(frame_cfg(w)) for _ in range(5)]
    rng = random.Random(7)
    for t in range(20):
        a.append_frames(sa, [t] * 5, w.frame_tokens)
        for s in sb:
            b.append_frame(s, t, w.frame_tokens)
        assert a.snapshot() == b.snapshot()
        for s in reversed(range(5)):
            if rng.random() < 0.5:
                a.rollback_last_frame(sa[s]); b.rollback_last_frame(sb[s])
        for s in range(5):
            if a.streams[sa[s]].undo is not None:
                a.evict_window(sa[s]); b.evict_window(sb[s])
        assert a.snapshot() == b.snapshot()
        check_pool(a)
    full = PagedCacheOracle(3, w.page_size)
    fs = [full.open_stream(frame_cfg(w)) for _ in range(2)]
    snap = full.snapshot()
    with pytest.raises(OracleError) as e:
        full.append_frames(fs, [0, 0], w.frame_tokens)     # needs 4 pages, 3 free
    assert e.value.code == "OOM"
    assert full.snapshot() == snap


def test_windowed_reset_carries_overlap():
    """Section 4: window_size counts KV slots (cached keyframes); when a window is
    full the cache resets and the last overlap keyframes carry over."""
    w = WORKLOADS["multistream"]
    o = PagedCacheOracle(w.pool_pages, w.page_size)
    sid = o.open_stream(frame_cfg(w))
    resets = 0
    for t in range(600):
        o.append_frame(sid, t, w.frame_tokens)
        st = o.streams[sid]
        assert st.kept <= w.window_slots
        o.evict_window(sid)
        if st.kept == w.overlap_keyframes and t > 8:
            resets += 1
            toks = o.visible_tokens(sid)
            frames = sorted({f for (_, f, _) in toks})
            assert frames == list(range(t - 7, t + 1))
            assert [p for p, _, _ in st.scale] == o.visible_table(sid)[0][:8]
            assert len(st.special) == 1 and st.sp_len == 48
        check_pool(o)
    # 128 slots per window, 8 carried: resets after keyframes 127, 247, 367, 487
    assert resets == 4


def test_close_stream_returns_everything():
    w = WORKLOADS["tiny"]
    o = PagedCacheOracle(w.pool_pages, w.page_size)
    sid = o.open_stream(frame_cfg(w))
    for t in range(9):
        o.append_frame(sid, t, w.frame_tokens)
        o.evict_window(sid)
    o.close_stream(sid)
    assert sorted(o.free) == list(range(w.pool_pages))
    c = o.open_stream(StreamConfig(mode="chunked", chunk_size=2, sliding_window_num=2,
                                   tokens_per_frame=20))
    for t in range(4):
        o.append_frame(c, t, 20)
        if t % 2 == 1:
            o.evict_window(c)
    o.append_frame(c, 4, 20)
    o.close_stream(c)
    assert sorted(o.free) == list(range(w.pool_pages))


def test_chunked_workload_shapes():
    """RFC section 2.3: sequence_length = sliding_window_num x chunk_size frames;
    a full chunk of 8 x 1374 tokens takes 43 pages (42 full + one of 240) and a
    chunk attends over 4 x 10,992 = 43,968 tokens."""
    w = WORKLOADS["chunked"]
    o = PagedCacheOracle(w.pool_pages, w.page_size)
    sid = o.open_stream(StreamConfig(mode="chunked", chunk_size=w.chunk_size,
                                     sliding_window_num=w.sliding_window_num,
                                     tokens_per_frame=w.tokens_per_frame))
    for c in range(6):
        for f in range(w.chunk_size):
            o.append_frame(sid, c * 8 + f, w.tokens_per_frame)
        idx, lens = o.visible_table(sid)
        assert o.current_chunk_tokens(sid) == 10992
        assert sum(lens) == 10992 * min(c + 1, 4)
        assert lens[:43] == [256] * 42 + [240]
        o.evict_window(sid)
        assert len(o.streams[sid].chunks) == min(c + 1, 3)
        check_pool(o)
