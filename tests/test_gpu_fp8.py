"""FP8 (E4M3) pages against the oracle (needs a GB300).

vLLM-Omni RFC "Reconstruction Engine", section 3.4 (quantization: KV cache
FP8). The stored codes and row exponents must equal the oracle's quantization
of the appended K/V bit for bit; the attention must match the fp64 oracle over
the dequantized K/V within the same tolerance as bf16 pages (the kernel computes
in bf16 on exactly those values)."""

import os
import random

import numpy as np
import pytest
import torch

from synth import TENSOR_K, WORKLOADS, is_keyframe
from tests.pairing import Pair, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_build_gb300 import build
    build.build()


def test_fp8_tiny_stream_every_frame():
    w = WORKLOADS["tiny"]
    pr = Pair(w, seed=0, fp8=True)
    sid = pr.open()
    for t in range(w.frames):
        pr.append(sid, t)
        pr.check_meta(sid)
        pr.check_pool(sid)
        out = pr.gpu.attend(pr.gpu_q_chunk(sid, 0, [t]), sid, 0, sm_scale=w.sm_scale)
        o, e = pr.oracle_attention(sid, 0, pr.cpu_q(sid, 0, [t]))
        assert_close(out, o, e, f"fp8 tiny frame {t}")
        pr.evict(sid)
    pr.gpu.sync()


def test_fp8_lingbot_stream_sampled_frames():
    """The one-layer LingBot-shaped stream on FP8 pages: tables on every frame,
    attention of every row at frames across the ramp and the steady state,
    codes and exponents of every visible slot at the end."""
    w = WORKLOADS["lingbot"]
    frames = int(os.environ.get("PKV_FP8_FRAMES", 300))
    pr = Pair(w, fp8=True)
    sid = pr.open()
    attend_at = {0, 8, 72, frames - 1}
    for t in range(frames):
        pr.append(sid, t)
        if t % 25 == 0:
            pr.check_meta(sid)
        if t in attend_at:
            out = pr.gpu.attend(pr.gpu_q_chunk(sid, 0, [t]), sid, 0, sm_scale=w.sm_scale)
            o, e = pr.oracle_attention(sid, 0, pr.cpu_q(sid, 0, [t]))
            assert_close(out, o, e, f"fp8 lingbot frame {t}")
        pr.evict(sid)
    pr.check_meta(sid)
    pr.check_pool(sid)
    pr.gpu.sync()


def test_fp8_long_stream_24_layers_keyframes():
    """The 24-layer keyframe stream (interval 4) on FP8 pages, its first 1,200
    frames: appends of every layer, rollbacks of non-keyframes; attention of
    two layers every 500 frames (every 8th row)."""
    w = WORKLOADS["long"]
    frames = int(os.environ.get("PKV_FP8_LONG_FRAMES", 1200))
    pr = Pair(w, fp8=True)
    sid = pr.open()
    rows = np.arange(0, w.frame_tokens, 8)
    for t in range(frames):
        pr.append(sid, t)
        if t % 50 == 0:
            pr.check_meta(sid)
        if t % 500 == 0 or t == frames - 1:
            for layer in (t // 500 % 24, 23):
                out = pr.gpu.attend(pr.gpu_q_chunk(sid, layer, [t]), sid, layer, sm_scale=w.sm_scale)
                o, e = pr.oracle_attention(sid, layer, pr.cpu_q(sid, layer, [t]), rows=rows)
                assert_close(out[torch.from_numpy(rows).cuda()], o, e, f"fp8 long frame {t} layer {layer}")
        if is_keyframe(t, w.num_scale, w.keyframe_interval):
            pr.evict(sid)
        else:
            pr.rollback(sid)
    pr.check_meta(sid)
    pr.check_pool(sid, layer=11)
    pr.gpu.sync()


@pytest.mark.parametrize("seed", [1, 3, 4])
def test_fp8_random_streams_with_windowed_resets(seed):
    """Small random shapes (page sizes 16..192, keyframes, rollbacks, windowed
    resets that copy carried rows between pages, two layers) on FP8 pages."""
    rng = random.Random(seed)
    ps = rng.choice([16, 32, 64, 128, 192])
    S = rng.randint(1, 3)
    w = WORKLOADS["tiny"].with_(page_size=ps, n_patch=ps, n_special=rng.randint(1, 6), num_scale=S,
                                window=rng.randint(1, 5), heads=rng.choice([1, 3, 4]),
                                window_slots=rng.randint(S + 1, 9), overlap_keyframes=rng.randint(0, S))
    pr = Pair(w, seed, layers=2, pool_pages=96, fp8=True)
    sid = pr.open()
    kf = rng.randint(1, 3)
    for t in range(rng.randint(20, 40)):
        pr.append(sid, t)
        pr.check_meta(sid)
        if t % 5 == 0:
            layer = t % 2
            pr.check_pool(sid, layer)
            out = pr.gpu.attend(pr.gpu_q_chunk(sid, layer, [t]), sid, layer, sm_scale=w.sm_scale)
            o, e = pr.oracle_attention(sid, layer, pr.cpu_q(sid, layer, [t]))
            assert_close(out, o, e, f"fp8 seed {seed} frame {t}")
        if is_keyframe(t, S, kf) and rng.random() > 0.15:
            pr.evict(sid)
        else:
            pr.rollback(sid)
        pr.check_meta(sid)
    pr.gpu.sync()


@pytest.mark.parametrize("ps", [16, 32])
def test_fp8_extra_rows_with_small_pages(ps):
    """Chunks of 2 frames of 131 tokens, i.e. 262 queries (two M-tiles plus extra
    rows, whose warps dequantize quarters of every tile), on FP8 pages of 16 and
    32 slots, so that a 64-slot tile spans four or two page blocks; 3 chunks
    visible, every row of every chunk."""
    w = WORKLOADS["chunked"].with_(page_size=ps, chunk_size=2, tokens_per_frame=131, sliding_window_num=3,
                                   heads=2, frames=10)
    pr = Pair(w, seed=5, fp8=True, pool_pages=128)
    sid = pr.open()
    for c in range(5):
        frames = [2 * c, 2 * c + 1]
        for f in frames:
            pr.append(sid, f)
        pr.check_meta(sid)
        out = pr.gpu.attend_chunked(pr.gpu_q_chunk(sid, 0, frames), sid, 0, sm_scale=w.sm_scale)
        o, e = pr.oracle_attention(sid, 0, pr.cpu_q(sid, 0, frames))
        assert_close(out, o, e, f"fp8 page {ps} chunk {c}")
        pr.evict(sid)
    pr.check_pool(sid)
    pr.gpu.sync()


def test_fp8_chunked_stream():
    """Chunked sliding-window attention on FP8 pages: chunks of 4 frames of 300
    tokens, 3 visible, 4 heads; every row of every chunk."""
    w = WORKLOADS["chunked"].with_(chunk_size=4, tokens_per_frame=300, sliding_window_num=3, heads=4,
                                   frames=24)
    pr = Pair(w, fp8=True, pool_pages=64)
    sid = pr.open()
    for c in range(6):
        frames = list(range(c * 4, c * 4 + 4))
        for f in frames:
            pr.append(sid, f)
        pr.check_meta(sid)
        q = pr.gpu_q_chunk(sid, 0, frames)
        out = pr.gpu.attend_chunked(q, sid, 0, sm_scale=w.sm_scale)
        o, e = pr.oracle_attention(sid, 0, pr.cpu_q(sid, 0, frames))
        assert_close(out, o, e, f"fp8 chunk {c}")
        pr.evict(sid)
    pr.check_pool(sid)
    pr.gpu.sync()


def test_fp8_batched_equals_separate_calls():
    w = WORKLOADS["lingbot"]
    pr = Pair(w, seed=2, pool_pages=512, fp8=True)
    lengths = [20, 75, 90]
    sids = [pr.open() for _ in lengths]
    for s, n in zip(sids, lengths):
        for t in range(n):
            pr.append(s, t)
            if t < n - 1:
                pr.evict(s)
    qs = [pr.gpu_q_chunk(s, 0, [n - 1]) for s, n in zip(sids, lengths)]
    outs = pr.gpu.attend_batched(qs, sids, 0, sm_scale=w.sm_scale)
    for s, q, out in zip(sids, qs, outs):
        single = pr.gpu.attend(q, s, 0, sm_scale=w.sm_scale)
        assert float((single.float() - out.float()).abs().max()) <= 2e-2
    pr.gpu.sync()


def test_fp8_pages_are_half_the_bytes_and_close_to_bf16():
    """The same frame on FP8 and bf16 pages: the FP8 result differs from the bf16
    one by the quantization alone (a few 2^-4-relative errors on K and V average
    out over ~19k slots), and both caches refuse the other's page reader."""
    from paged_kv_cache_build_gb300 import PkvError
    w = WORKLOADS["lingbot"]
    a, b = Pair(w, fp8=True), Pair(w)
    sa, sb = a.open(), b.open()
    for t in range(100):
        for pr, s in ((a, sa), (b, sb)):
            pr.append(s, t)
            if t < 99:
                pr.evict(s)
    q = a.gpu_q_chunk(sa, 0, [99])
    oa = a.gpu.attend(q, sa, 0, sm_scale=w.sm_scale).float()
    ob = b.gpu.attend(q, sb, 0, sm_scale=w.sm_scale).float()
    d = (oa - ob).abs()
    assert float(d.max()) < 0.05 and float(d.mean()) < 5e-3, (float(d.max()), float(d.mean()))
    with pytest.raises(PkvError):
        a.gpu.read_page(0, 0)
    with pytest.raises(PkvError):
        b.gpu.read_page_fp8(0, 0)
    k = a.gpu_tensor(sa, 0, 100, TENSOR_K)
    with pytest.raises(PkvError):
        a.gpu.attend_blocksparse(q, sa, 0, keep=4)
    del k
    a.gpu.sync()
    b.gpu.sync()
