"""pkv_stream_frames: a run of frames driven from native code equals the same
frames as separate pkv_append_frame / pkv_attend / pkv_evict_window or
pkv_rollback_last_frame calls ("LingBot-Map Paged KV Cache", sections 2-3):
bit-identical outputs, page tables and free stacks."""

import numpy as np
import pytest
import torch

from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS, is_keyframe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_build_gb300 import build
    build.build()


def _inputs(w, n):
    from paged_kv_cache_build_gb300 import synth_fill
    shape = (n, w.frame_tokens, w.heads, w.head_dim)
    q, k, v = (torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(3))
    synth_fill(q, 3, w.index, 0, 0, 0, TENSOR_Q, 0, w.q_scale)
    synth_fill(k, 3, w.index, 0, 0, 0, TENSOR_K)
    synth_fill(v, 3, w.index, 0, 0, 0, TENSOR_V)
    return q, k, v


def _pair(w, pool_pages=None):
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg
    caches, sids = [], []
    for _ in range(2):
        c = PagedKVCache(pool_pages or w.pool_pages, w.page_size, w.heads, w.head_dim)
        caches.append(c)
        sids.append(c.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special)))
    return caches, sids


def _state(c, sid):
    idx, lens, n, last = c.build_visible_page_table(sid)
    k = int(n.item())
    return idx.cpu().numpy()[:k].tolist(), lens.cpu().numpy()[:k].tolist(), c.free_pages()


@pytest.mark.parametrize("name,frames,interval", [("lingbot", 100, 1), ("tiny", 12, 1),
                                                  ("lingbot", 90, 4)])
def test_run_equals_separate_calls(name, frames, interval):
    w = WORKLOADS[name]
    q, k, v = _inputs(w, frames)
    (a, b), (sa, sb) = _pair(w)
    keys = [is_keyframe(t, w.num_scale, interval) for t in range(frames)]
    out_a = torch.empty_like(q)
    # native runs of uneven length
    t0 = 0
    for n in (7, 30, frames):
        t1 = min(frames, t0 + n)
        a.stream_frames(sa, q[t0:t1], k[t0:t1], v[t0:t1], keyframe=keys[t0:t1] if interval > 1 else None,
                        out=out_a[t0:t1], sm_scale=w.sm_scale)
        t0 = t1
    out_b = torch.empty_like(q)
    for t in range(frames):
        b.append_frame(sb, k[t], v[t])
        b.attend(q[t], sb, out=out_b[t], sm_scale=w.sm_scale)
        if keys[t]:
            b.evict_window(sb)
        else:
            b.rollback_last_frame(sb)
    assert torch.equal(out_a, out_b)
    assert _state(a, sa) == _state(b, sb)
    a.sync()
    b.sync()


def test_errors_and_partial_runs():
    from paged_kv_cache_build_gb300 import PkvError, chunked_stream_cfg
    w = WORKLOADS["tiny"]
    q, k, v = _inputs(w, 12)
    (a, b), (sa, sb) = _pair(w, pool_pages=9)
    z = q[:0]
    assert a.stream_frames(sa, z, z, z).shape == z.shape                  # no frames: a no-op
    with pytest.raises(PkvError) as ei:                                    # wrong token count
        a.stream_frames(sa, q[:, :10].contiguous(), k[:, :10].contiguous(), v[:, :10].contiguous())
    assert ei.value.code == "INVALID"
    a.append_frame(sa, k[0], v[0])                                          # a pending frame
    with pytest.raises(PkvError) as ei:
        a.stream_frames(sa, q[:2], k[:2], v[:2])
    assert ei.value.code == "STATE"
    a.rollback_last_frame(sa)
    cid = a.open_stream(chunked_stream_cfg(2, 2, w.frame_tokens))
    with pytest.raises(PkvError) as ei:
        a.stream_frames(cid, q[:2], k[:2], v[:2])
    assert ei.value.code == "STATE"
    a.close_stream(cid)
    # a pool too small for the run: the frames before the failing one stay applied
    with pytest.raises(PkvError) as ei:
        a.stream_frames(sa, q, k, v, sm_scale=w.sm_scale)
    assert ei.value.code == "OOM" and "frame " in str(ei.value)
    failed = int(str(ei.value).split("frame ")[1].split(":")[0])
    for t in range(failed):
        b.append_frame(sb, k[t], v[t])
        b.attend(q[t], sb, sm_scale=w.sm_scale)
        b.evict_window(sb)
    assert _state(a, sa) == _state(b, sb)
    a.sync()
    b.sync()


@pytest.mark.parametrize("fp8", [False, True])
def test_multi_layer_run_equals_separate_calls(fp8):
    """pkv_stream_frames_multi: 3 layers, a ring of 5 input frames, keyframe
    interval 4 (rollbacks), frame events; equal to the separate per-layer calls."""
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    w = WORKLOADS["long"]
    L, R, frames = 3, 5, 90
    shape = (L, R, w.frame_tokens, w.heads, w.head_dim)
    q, k, v = (torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(3))
    for layer in range(L):
        synth_fill(q[layer], 1, w.index, 0, layer, 0, TENSOR_Q, 0, w.q_scale)
        synth_fill(k[layer], 1, w.index, 0, layer, 0, TENSOR_K)
        synth_fill(v[layer], 1, w.index, 0, layer, 0, TENSOR_V)
    caches = [PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim, layers=L, fp8=fp8)
              for _ in range(2)]
    sids = [c.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
            for c in caches]
    keys = [is_keyframe(t, w.num_scale, 4) for t in range(frames)]
    out_a = torch.zeros_like(q)
    out_b = torch.zeros_like(q)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(41)]
    caches[0].stream_frames_multi(sids[0], list(q), list(k), list(v), list(out_a), 0, 40, keys[:40],
                                  sm_scale=w.sm_scale, events=events)
    caches[0].stream_frames_multi(sids[0], list(q), list(k), list(v), list(out_a), 40, 50, keys[40:],
                                  sm_scale=w.sm_scale)
    b, sb = caches[1], sids[1]
    for t in range(frames):
        for layer in range(L):
            b.append_frame(sb, k[layer, t % R], v[layer, t % R], layer)
            b.attend(q[layer, t % R], sb, layer, out=out_b[layer, t % R], sm_scale=w.sm_scale)
        if keys[t]:
            b.evict_window(sb)
        else:
            b.rollback_last_frame(sb)
    torch.cuda.synchronize()
    assert all(events[i].elapsed_time(events[i + 1]) > 0 for i in range(40))
    np.testing.assert_array_equal(out_a.view(torch.int16).cpu().numpy(), out_b.view(torch.int16).cpu().numpy())
    assert _state(caches[0], sids[0]) == _state(b, sb)
    for c in caches:
        c.sync()
        c.close()


def test_model_run_equals_separate_calls():
    """pkv_stream_model_frames: 3 layers, a ring of 5 input frames, keyframe
    interval 4; each layer's frame attention, append and global attention equal
    the same calls made one by one, outputs bit for bit and the cache state."""
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    w = WORKLOADS["long"]
    L, R, frames = 3, 5, 30
    shape = (L, R, w.frame_tokens, w.heads, w.head_dim)
    q, k, v, fq, fk, fv = (torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(6))
    for layer in range(L):
        synth_fill(q[layer], 2, w.index, 0, layer, 0, TENSOR_Q, 0, w.q_scale)
        synth_fill(k[layer], 2, w.index, 0, layer, 0, TENSOR_K)
        synth_fill(v[layer], 2, w.index, 0, layer, 0, TENSOR_V)
        synth_fill(fq[layer], 3, w.index, 0, layer, 0, TENSOR_Q, 0, w.q_scale)
        synth_fill(fk[layer], 3, w.index, 0, layer, 0, TENSOR_K)
        synth_fill(fv[layer], 3, w.index, 0, layer, 0, TENSOR_V)
    caches = [PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim, layers=L) for _ in range(2)]
    sids = [c.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
            for c in caches]
    keys = [is_keyframe(t, w.num_scale, 4) for t in range(frames)]
    out_a, fout_a = torch.zeros_like(q), torch.zeros_like(q)
    out_b, fout_b = torch.zeros_like(q), torch.zeros_like(q)
    caches[0].stream_model_frames(sids[0], list(fq), list(fk), list(fv), list(fout_a), list(q), list(k),
                                  list(v), list(out_a), 0, frames, keys, sm_scale=w.sm_scale)
    b, sb = caches[1], sids[1]
    for t in range(frames):
        for layer in range(L):
            b.attend_frames(fq[layer, t % R], fk[layer, t % R], fv[layer, t % R],
                            out=fout_b[layer, t % R], sm_scale=w.sm_scale)
            b.append_frame(sb, k[layer, t % R], v[layer, t % R], layer)
            b.attend(q[layer, t % R], sb, layer, out=out_b[layer, t % R], sm_scale=w.sm_scale)
        if keys[t]:
            b.evict_window(sb)
        else:
            b.rollback_last_frame(sb)
    torch.cuda.synchronize()
    for got, want in ((out_a, out_b), (fout_a, fout_b)):
        np.testing.assert_array_equal(got.view(torch.int16).cpu().numpy(), want.view(torch.int16).cpu().numpy())
    assert _state(caches[0], sids[0]) == _state(b, sb)
    from paged_kv_cache_build_gb300._lib import STATUS_NAMES
    status = caches[0].lib.pkv_stream_model_frames(caches[0].h, sids[0], L, None, None, None, None,
                                                   None, None, None, None, R, frames, 1, w.frame_tokens,
                                                   None, 0.0, None, None)
    assert STATUS_NAMES.get(status) == "INVALID"                 # null frame-attention rings
    for c in caches:
        c.sync()
        c.close()
