"""The five synthetic workloads, as shapes and call schedules.

W0  tiny stream: 12 frames of 16 patch + 6 special tokens, page_size 16,
    2 scale frames, 4-frame window, 4 heads x 64, keyframe interval 1.
W1  LingBot-Map-shaped stream, one layer: 512 frames of 256 patch + 6
    special tokens, page_size 256, 8 scale frames, 64-frame window,
    16 heads x 64, queries ~N(0,1)/8.
W2  the W1 shapes with 24 layers (one page set per layer, one shared page
    table), 10,000 frames, keyframe interval 4.
W3  VGGT-style chunked sliding-window global attention: 1374 tokens per
    frame, 8-frame chunks, 4 chunks visible, 16 heads x 64, 64 chunks.
W4  32 streams sharing one pool, lengths uniform in [100, 5000], keyframe
    interval drawn from {1, 2, 4, 8}, W1 shapes, windowed mode with 128 KV
    slots per window and 8 overlap keyframes.

The keyframe schedule is the caller's policy, not the cache's: frame t is a
keyframe when t < num_scale or (t - num_scale) is a multiple of the
interval, so scale frames are always kept.
"""

from dataclasses import dataclass, field, replace
from typing import Tuple

from .inputs import uniform_draw


@dataclass(frozen=True)
class Workload:
    name: str
    index: int                 # workload field of the generator key
    mode: str                  # "frame" or "chunked"
    frames: int                # frames per stream (chunked: chunks * chunk_size)
    page_size: int
    heads: int = 16
    head_dim: int = 64
    layers: int = 1
    pool_pages: int = 128
    q_scale: float = 1.0       # power of two applied to generated queries
    # frame mode
    n_patch: int = 0
    n_special: int = 0
    num_scale: int = 0
    window: int = 0
    keyframe_interval: int = 1
    window_slots: int = 0
    overlap_keyframes: int = 0
    streams: int = 1
    # chunked mode
    tokens_per_frame: int = 0
    chunk_size: int = 0
    sliding_window_num: int = 0
    extra: Tuple = field(default=())

    @property
    def frame_tokens(self):
        return self.n_patch + self.n_special if self.mode == "frame" else self.tokens_per_frame

    @property
    def sm_scale(self):
        return self.head_dim ** -0.5

    def with_(self, **kw):
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload(name="tiny", index=0, mode="frame", frames=12, page_size=16, heads=4,
                     pool_pages=64, n_patch=16, n_special=6, num_scale=2, window=4),
    "lingbot": Workload(name="lingbot", index=1, mode="frame", frames=512, page_size=256,
                        pool_pages=128, q_scale=0.125, n_patch=256, n_special=6,
                        num_scale=8, window=64),
    "long": Workload(name="long", index=2, mode="frame", frames=10000, page_size=256,
                     layers=24, pool_pages=160, q_scale=0.125, n_patch=256, n_special=6,
                     num_scale=8, window=64, keyframe_interval=4),
    "chunked": Workload(name="chunked", index=3, mode="chunked", frames=64 * 8, page_size=256,
                        pool_pages=192, tokens_per_frame=1374, chunk_size=8,
                        sliding_window_num=4),
    "multistream": Workload(name="multistream", index=4, mode="frame", frames=5000,
                            page_size=256, pool_pages=4096, q_scale=0.125, n_patch=256,
                            n_special=6, num_scale=8, window=64, window_slots=128,
                            overlap_keyframes=8, streams=32),
}


def is_keyframe(t, num_scale, interval):
    """Caller-side keyframe policy (scale frames are always kept)."""
    return t < num_scale or (t - num_scale) % interval == 0


def multistream_schedule(seed, workload=WORKLOADS["multistream"], lo=100, hi=5000):
    """Per-stream (length, keyframe interval) for the shared-pool workload,
    drawn from the counter-based generator."""
    out = []
    for s in range(workload.streams):
        length = lo + uniform_draw(seed, workload.index, s, 0) % (hi - lo + 1)
        interval = (1, 2, 4, 8)[uniform_draw(seed, workload.index, s, 1) % 4]
        out.append((length, interval))
    return out
