"""pkv_attend_noalloc: the attention call for callers that cannot allocate device
memory when they call it (for example while a CUDA graph is being captured, or in
a frame loop that cannot afford cudaMalloc's device-wide synchronisation). Its
split-KV partials live in a fixed device array compiled into the library.

Checked through the C ABI against pkv_attend on the same stream, twice in a row
(the array keeps the previous call's contents), and for the size limit. This file
is collected last; it builds the library itself, so it also runs on its own."""

import ctypes

import numpy as np
import pytest
import torch

from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2     # the tolerance the parity tests use
MEAN_ABS = 2e-3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_build_gb300 import build
    from paged_kv_cache_build_gb300._lib import load
    build.build()
    return load()


def _fill(t, w, sid, frame, tensor, scale=1.0):
    from paged_kv_cache_build_gb300 import synth_fill
    return synth_fill(t, 0, w.index, sid, 0, frame, tensor, 0, scale)


def _noalloc(lib, cache, q, sid, out, sm_scale):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pkv_attend_noalloc(cache.h, ctypes.c_void_p(q.data_ptr()), q.shape[0], sid, 0,
                                  ctypes.c_void_p(out.data_ptr()), ctypes.c_float(sm_scale), stream)


def _close(a, b):
    d = (a.float() - b.float()).abs()
    return float(d.max()), float(d.mean())


@pytest.mark.parametrize("name,frames", [("tiny", 12), ("lingbot", 120)])
def test_noalloc_matches_attend_twice(lib, name, frames):
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg
    w = WORKLOADS[name]
    cache = PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim)
    sid = cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
    shape = (w.frame_tokens, w.heads, w.head_dim)
    k = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    q = torch.empty_like(k)
    for t in range(frames):
        _fill(k, w, sid, t, TENSOR_K)
        _fill(v, w, sid, t, TENSOR_V)
        cache.append_frame(sid, k, v)
        if t % 40 == 39 or t == frames - 1:
            _fill(q, w, sid, t, TENSOR_Q, w.q_scale)
            ref = cache.attend(q, sid, sm_scale=w.sm_scale)
            for _ in range(2):                       # two calls in a row
                got = torch.full_like(q, float("nan"))
                assert _noalloc(lib, cache, q, sid, got, w.sm_scale) == 0, lib.pkv_last_error(cache.h)
                torch.cuda.synchronize()
                mx, mean = _close(got, ref)
                assert mx <= MAX_ABS and mean <= MEAN_ABS, (mx, mean)
                assert torch.isfinite(got.float()).all()
        cache.evict_window(sid)
    cache.sync()
    cache.close()


def test_noalloc_rejects_more_than_its_scratch(lib):
    """A whole chunk of 8 x 1374 queries over the full window of 4 chunks (687
    tiles, 3 KV splits) needs more split-KV scratch than the fixed 16 MiB: the
    call refuses, launches nothing, and pkv_attend still works."""
    from paged_kv_cache_build_gb300 import PagedKVCache, chunked_stream_cfg
    w = WORKLOADS["chunked"]
    cache = PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim)
    sid = cache.open_stream(chunked_stream_cfg(w.chunk_size, w.sliding_window_num, w.tokens_per_frame))
    kv = torch.empty((w.chunk_size, w.tokens_per_frame, w.heads, w.head_dim), dtype=torch.bfloat16,
                     device="cuda")
    _fill(kv, w, sid, 0, TENSOR_K)
    for c in range(w.sliding_window_num):
        for f in range(w.chunk_size):
            cache.append_frame(sid, kv[f], kv[f])
        if c < w.sliding_window_num - 1:
            cache.evict_window(sid)
    n_q = w.chunk_size * w.tokens_per_frame
    q = torch.zeros((n_q, w.heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    # whole-chunk attention runs in several KV splits: 3 x 10,992 x 16 x 264 bytes > 16 MiB
    assert _noalloc(lib, cache, q, sid, out, w.sm_scale) == 1
    assert b"static scratch" in lib.pkv_last_error(cache.h)
    ref = cache.attend_chunked(q, sid, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert torch.isfinite(ref.float()).all()
    cache.sync()
    cache.close()


def test_noalloc_chunked_uses_the_static_scratch(lib):
    """A small chunked stream (chunks of 2 x 400 tokens, 4 visible, 4 heads,
    64-slot pages) whose whole-chunk call fits the fixed array: every call runs in
    several KV splits (two launches: the attention and the combine that reads the
    partials back from the array) and matches pkv_attend_chunked, twice in a row."""
    from paged_kv_cache_build_gb300 import PagedKVCache, chunked_stream_cfg, kernel_launches
    w = WORKLOADS["chunked"]
    heads, tokens, chunk, window = 4, 400, 2, 4
    cache = PagedKVCache(128, 64, heads, 64)
    sid = cache.open_stream(chunked_stream_cfg(chunk, window, tokens))
    kv = torch.empty((2, chunk, tokens, heads, 64), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((chunk * tokens, heads, 64), dtype=torch.bfloat16, device="cuda")
    for c in range(6):
        _fill(kv[0], w, sid, c * chunk, TENSOR_K)
        _fill(kv[1], w, sid, c * chunk, TENSOR_V)
        _fill(q.view(chunk, tokens, heads, 64), w, sid, c * chunk, TENSOR_Q)
        for f in range(chunk):
            cache.append_frame(sid, kv[0, f], kv[1, f])
        ref = cache.attend_chunked(q, sid, sm_scale=w.sm_scale)
        torch.cuda.synchronize()
        for _ in range(2):
            got = torch.full_like(q, float("nan"))
            n0 = kernel_launches()
            assert _noalloc(lib, cache, q, sid, got, w.sm_scale) == 0, lib.pkv_last_error(cache.h)
            assert kernel_launches() - n0 == 2          # split: attention + combine
            torch.cuda.synchronize()
            mx, mean = _close(got, ref)
            assert mx <= MAX_ABS and mean <= MEAN_ABS, (c, mx, mean)
            assert torch.isfinite(got.float()).all()
        cache.evict_window(sid)
    cache.sync()
    cache.close()
