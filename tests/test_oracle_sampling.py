"""Pins of the oracle's per-layer random page subset (oracle/sampling.py): its
splitmix64 against the published sequence, the two limits that reduce it to a
plain definition (keep everything: the visible tokens; keep nothing: the scale
pages), and the binomial statistics of the keep rule."""

import math

from oracle import PagedCacheOracle, StreamConfig
from oracle.sampling import kept_positions, page_kept, splitmix64


def test_splitmix64_published_sequence():
    # splitmix64 seeded with 1234567: each output advances the state by the
    # golden gamma, then mixes; the first five published outputs
    expected = [6457827717110365317, 3203168211198807973, 9817491932198370423,
                4593380528125082431, 16408922859458223821]
    gamma = 0x9E3779B97F4A7C15
    assert [splitmix64((1234567 + i * gamma) % (1 << 64)) for i in range(5)] == expected


def _stream(frames=90):
    ora = PagedCacheOracle(256, 256, 4)
    sid = ora.open_stream(StreamConfig(mode="frame", num_scale=8, window=64, n_patch=256, n_special=6))
    for t in range(frames):
        ora.append_frame(sid, t, 262)
        if t < frames - 1:
            ora.evict_window(sid)
    return ora, sid


def test_keep_all_is_the_visible_tokens_and_keep_none_the_anchors():
    ora, sid = _stream()
    assert ora.visible_tokens_sampled(sid, 7, 3, 65536) == ora.visible_tokens(sid)
    idx, lens = ora.visible_table(sid)
    anchors = []
    for p, n in zip(idx[:8], lens[:8]):
        anchors.extend(ora.slots[p][:n])
    assert ora.visible_tokens_sampled(sid, 7, 3, 0) == anchors
    assert all(f < 8 for _, f, _ in anchors)                 # the scale frames


def test_keep_rule_statistics_and_layer_independence():
    n, keep = 20000, 16384                                   # keep one in four
    for layer in (0, 1, 23):
        kept = sum(page_kept(12345, layer, e, keep) for e in range(n))
        # binomial(n, 1/4): mean 5000, sd ~61; six sd either side
        assert abs(kept - n / 4) < 6 * math.sqrt(n * 0.25 * 0.75)
    a = [page_kept(12345, 0, e, keep) for e in range(n)]
    b = [page_kept(12345, 1, e, keep) for e in range(n)]
    both = sum(x and y for x, y in zip(a, b))
    # independent layers: P(both) = 1/16
    assert abs(both - n / 16) < 6 * math.sqrt(n / 16 * 15 / 16)
    c = [page_kept(54321, 0, e, keep) for e in range(n)]
    assert a != c                                            # the seed matters


def test_kept_positions_keeps_anchors_and_table_order():
    pos = kept_positions(80, 8, 99, 5, 30000)
    assert pos[:8] == list(range(8))
    assert pos == sorted(set(pos))
    assert all(page_kept(99, 5, e, 30000) for e in pos[8:])
    assert all(e in pos for e in range(8, 80) if page_kept(99, 5, e, 30000))
