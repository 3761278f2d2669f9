"""Host-side behaviour of the library that needs a device: call-order refusals
that change nothing, and the split-KV scratch that pkv_stream_open sizes up front
so that the attention calls of a stream never allocate or synchronise (needs a
GB300)."""

import numpy as np
import pytest
import torch

from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS
from tests.pairing import Pair

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_build_gb300 import build
    build.build()


def test_append_while_a_frame_is_pending_is_refused():
    """"LingBot-Map Paged KV Cache", section 3: a frame is appended, attended,
    then either rolled back or committed. A second layer-0 append before either
    would silently commit the first frame past the window's accounting, so it
    is refused (STATE) and changes nothing; after the rollback it goes through."""
    from paged_kv_cache_build_gb300 import PkvError
    w = WORKLOADS["tiny"]
    pr = Pair(w)
    sid = pr.open()
    for t in range(5):
        pr.append(sid, t)
        pr.evict(sid)
    pr.append(sid, 5)
    before = pr.gpu.export_state(sid)
    k = pr.gpu_tensor(sid, 0, 6, TENSOR_K)
    with pytest.raises(PkvError) as e:
        pr.gpu.append_frame(sid, k, k)
    assert e.value.code == "STATE" and "pending" in str(e.value)
    with pytest.raises(PkvError) as e:
        pr.gpu.append_frames([sid], [k], [k])
    assert e.value.code == "STATE"
    assert pr.gpu.export_state(sid) == before
    pr.rollback(sid)
    pr.append(sid, 6)
    pr.check_meta(sid)
    pr.evict(sid)
    pr.check_meta(sid)
    pr.gpu.sync()


def test_stream_open_sizes_the_scratch_for_the_whole_stream():
    """After pkv_stream_open, the 512-frame LingBot-shaped stream's attention
    calls (every table size from 1 to 85 pages) never reallocate the scratch."""
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    w = WORKLOADS["lingbot"]
    cache = PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim)
    assert cache.scratch_info() == (0, 0)
    sid = cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
    nbytes, allocs = cache.scratch_info()
    assert allocs == 1 and nbytes > 0
    R = 4
    x = torch.empty((3, R, w.frame_tokens, w.heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    synth_fill(x[0], 0, w.index, sid, 0, 0, TENSOR_Q, 0, w.q_scale)
    synth_fill(x[1], 0, w.index, sid, 0, 0, TENSOR_K)
    synth_fill(x[2], 0, w.index, sid, 0, 0, TENSOR_V)
    out = torch.empty_like(x[0, 0])
    for t in range(w.frames):
        cache.append_frame(sid, x[1, t % R], x[2, t % R])
        cache.attend(x[0, t % R], sid, out=out, sm_scale=w.sm_scale)
        cache.evict_window(sid)
    cache.sync()
    assert cache.scratch_info() == (nbytes, 1)
    cache.close()


def test_first_attend_of_a_long_stream_can_be_graph_captured():
    """A stream that has never attended, 100 frames long: its first pkv_attend is
    captured into a CUDA graph (a capture fails on any device-wide synchronisation)
    and the replay equals the eager call bit for bit."""
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    w = WORKLOADS["lingbot"]
    cache = PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim)
    sid = cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
    kv = torch.empty((2, w.frame_tokens, w.heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    for t in range(100):
        synth_fill(kv[0], 0, w.index, sid, 0, t, TENSOR_K)
        synth_fill(kv[1], 0, w.index, sid, 0, t, TENSOR_V)
        cache.append_frame(sid, kv[0], kv[1])
        if t < 99:
            cache.evict_window(sid)
    q = torch.empty((w.frame_tokens, w.heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    synth_fill(q, 0, w.index, sid, 0, 99, TENSOR_Q, 0, w.q_scale)
    out_g = torch.full_like(q, float("nan"))
    torch.cuda.synchronize()
    allocs = cache.scratch_info()[1]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            cache.attend(q, sid, out=out_g, sm_scale=w.sm_scale, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    ref = cache.attend(q, sid, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert cache.scratch_info()[1] == allocs
    np.testing.assert_array_equal(out_g.view(torch.int16).cpu().numpy(),
                                  ref.view(torch.int16).cpu().numpy())
    cache.sync()
    cache.close()
