"""pkv_attend_frames (intra-frame attention, vLLM-Omni RFC "Reconstruction
Engine", sections 2.2 and 3.3) against the fp64 oracle: every frame's tokens over
that frame's own tokens, K and V read through TMA tensor maps. Sizes span one
and several M-groups, the extra-row shapes, ragged last tiles and frames that
end inside a tile shared with the next frame."""

import numpy as np
import pytest
import torch

from oracle import frame_attend_fp64
from synth import TENSOR_K, TENSOR_Q, TENSOR_V, frame_tensor
from tests.pairing import assert_close

pytestmark = pytest.mark.gpu

WL = 5          # generator workload index used by these cases


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_build_gb300 import build
    build.build()


def _inputs(seed, F, T, H, q_scale=0.125):
    from paged_kv_cache_build_gb300 import synth_fill
    dev = {}
    host = {}
    for name, tensor, scale in (("q", TENSOR_Q, q_scale), ("k", TENSOR_K, 1.0), ("v", TENSOR_V, 1.0)):
        t = torch.empty((F, T, H, 64), dtype=torch.bfloat16, device="cuda")
        synth_fill(t, seed, WL, 0, 0, 0, tensor, 0, scale)
        dev[name] = t
        host[name] = np.stack([frame_tensor(seed, WL, 0, 0, f, tensor, T, H, 64, scale) for f in range(F)])
    return dev, host


def _oracle(host, sm_scale):
    o = frame_attend_fp64(host["q"], host["k"], host["v"], sm_scale)
    e = frame_attend_fp64(host["q"], host["k"], host["v"] & np.uint16(0x7FFF), sm_scale)
    return o, e


CASES = [  # (frames, tokens, heads)
    (1, 262, 16),     # a LingBot-Map frame: two M-tiles + 6 extra rows
    (3, 22, 4),       # the tiny workload's frame
    (2, 1374, 16),    # a VGGT frame: six M-groups, 22 tiles, ragged last tile
    (4, 1, 2),
    (2, 64, 2),
    (2, 65, 2),
    (1, 128, 4),
    (2, 136, 4),      # one M-tile + 8 extra rows
    (2, 137, 4),      # two M-tiles
    (3, 257, 2),
    (1, 264, 4),      # two M-tiles + 8 extra rows
    (2, 265, 2),      # two M-groups
    (1, 600, 3),
]


@pytest.mark.parametrize("F,T,H", CASES)
def test_frames_against_oracle(F, T, H):
    from paged_kv_cache_build_gb300 import PagedKVCache
    c = PagedKVCache(4, 16, H)
    dev, host = _inputs((7 * F + T) % 97, F, T, H)
    out = c.attend_frames(dev["q"], dev["k"], dev["v"], sm_scale=0.125)
    o, e = _oracle(host, 0.125)
    assert_close(out, o, e, f"{F} frames x {T} tokens x {H} heads")
    c.sync()
    c.close()


def test_default_scale_and_single_frame_layout():
    """sm_scale <= 0 means 1/sqrt(64); a [tokens][heads][64] tensor is one frame."""
    from paged_kv_cache_build_gb300 import PagedKVCache
    c = PagedKVCache(4, 16, 4)
    dev, host = _inputs(11, 1, 70, 4, q_scale=1.0)
    out = c.attend_frames(dev["q"][0], dev["k"][0], dev["v"][0])
    o, e = _oracle(host, 0.125)
    assert_close(out[None], o, e, "default scale")
    c.sync()
    c.close()


def test_batch_equals_separate_frames():
    """Frames in one launch give bit-identical results to one call per frame."""
    from paged_kv_cache_build_gb300 import PagedKVCache
    c = PagedKVCache(4, 16, 16)
    dev, _ = _inputs(3, 4, 262, 16)
    together = c.attend_frames(dev["q"], dev["k"], dev["v"], sm_scale=0.125)
    for f in range(4):
        alone = c.attend_frames(dev["q"][f], dev["k"][f], dev["v"][f], sm_scale=0.125)
        assert torch.equal(alone, together[f])
    c.sync()
    c.close()


def test_a_frame_ignores_the_others():
    """Replacing one frame's K and V changes only that frame's output."""
    from paged_kv_cache_build_gb300 import PagedKVCache, synth_fill
    c = PagedKVCache(4, 16, 4)
    dev, _ = _inputs(4, 3, 150, 4)
    base = c.attend_frames(dev["q"], dev["k"], dev["v"], sm_scale=0.125)
    k2, v2 = dev["k"].clone(), dev["v"].clone()
    synth_fill(k2[1], 99, WL, 1, 0, 0, TENSOR_K)
    synth_fill(v2[1], 99, WL, 1, 0, 0, TENSOR_V)
    moved = c.attend_frames(dev["q"], k2, v2, sm_scale=0.125)
    assert torch.equal(moved[0], base[0]) and torch.equal(moved[2], base[2])
    assert not torch.equal(moved[1], base[1])
    c.sync()
    c.close()


def test_errors_and_empty_batch():
    from paged_kv_cache_build_gb300 import PagedKVCache, PkvError
    c = PagedKVCache(4, 16, 2)
    z = torch.zeros((0, 10, 2, 64), dtype=torch.bfloat16, device="cuda")
    assert c.attend_frames(z, z, z).shape == z.shape            # no frames: a no-op
    flat = torch.zeros(2 * 10 * 2 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    odd = flat[1:1 + 2 * 10 * 2 * 64].view(2, 10, 2, 64)       # 2-byte offset: unaligned
    good = torch.zeros((2, 10, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(PkvError) as ei:
        c.attend_frames(odd, good, good)
    assert ei.value.code == "INVALID"
    with pytest.raises(PkvError):
        c.attend_frames(good, odd, good)
    with pytest.raises(ValueError):
        c.attend_frames(good, good[:1], good)
    with pytest.raises(ValueError):
        c.attend_frames(torch.zeros((2, 10, 3, 64), dtype=torch.bfloat16, device="cuda"),
                        torch.zeros((2, 10, 3, 64), dtype=torch.bfloat16, device="cuda"),
                        torch.zeros((2, 10, 3, 64), dtype=torch.bfloat16, device="cuda"))
    c.sync()
    c.close()
