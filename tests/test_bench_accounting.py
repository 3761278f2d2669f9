"""The benchmark's FLOP accounting: its closed form for the visible tokens of
frame t must equal the cache oracle's count for every frame of the LingBot-shaped
stream (and of the tiny one), so the reported TFLOP/s counts exactly the useful
work (4 * n_q * N_kv * 64 per head)."""

import bench
from oracle import PagedCacheOracle, StreamConfig
from synth import WORKLOADS


def _oracle_counts(w):
    ora = PagedCacheOracle(w.pool_pages, w.page_size)
    sid = ora.open_stream(StreamConfig(mode="frame", num_scale=w.num_scale, window=w.window,
                                       n_patch=w.n_patch, n_special=w.n_special))
    out = []
    for t in range(w.frames):
        ora.append_frame(sid, t, w.frame_tokens)
        out.append(len(ora.visible_tokens(sid)))
        ora.evict_window(sid)
    return out


def test_visible_tokens_closed_form():
    for name in ("lingbot", "tiny"):
        w = WORKLOADS[name]
        counts = _oracle_counts(w)
        assert [bench.visible_tokens(w, t) for t in range(w.frames)] == counts
    w = WORKLOADS["lingbot"]
    assert bench.visible_tokens(w, 511) == 21504          # 8*256 + 64*256 + 512*6


def test_frame_flops():
    w = WORKLOADS["lingbot"]
    assert bench.frame_flops(w, 21504) == 4.0 * 262 * 21504 * 64 * 16
