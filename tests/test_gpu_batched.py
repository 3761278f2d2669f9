"""pkv_attend_batched: several streams' attention in one launch (LingBot-Map
Paged KV Cache, section 4's multi-stream pool), against the fp64 oracle and
against the same streams' separate pkv_attend calls."""

import numpy as np
import pytest
import torch

from tests.pairing import Pair, assert_close
from synth import WORKLOADS

pytestmark = pytest.mark.gpu


def _streams(pr, lengths):
    """Open one stream per length and append that many frames to it (keyframes
    throughout: the window is evicted after every frame but the last)."""
    sids = [pr.open() for _ in lengths]
    for s, n in zip(sids, lengths):
        for t in range(n):
            pr.append(s, t)
            if t < n - 1:
                pr.evict(s)
    return sids


def test_batched_tiny_streams_match_oracle_and_separate_calls():
    w = WORKLOADS["tiny"]
    pr = Pair(w, seed=1, layers=1)
    lengths = [1, 3, 5, 7, 9]
    sids = _streams(pr, lengths)
    qs = [pr.gpu_q_chunk(s, 0, [n - 1]) for s, n in zip(sids, lengths)]
    outs = pr.gpu.attend_batched(qs, sids, 0, sm_scale=w.sm_scale)
    for s, n, q, out in zip(sids, lengths, qs, outs):
        o, e = pr.oracle_attention(s, 0, pr.cpu_q(s, 0, [n - 1]))
        assert_close(out, o, e, f"batched stream {s}")
        single = pr.gpu.attend(q, s, 0, sm_scale=w.sm_scale)
        assert_close(single, o, e, f"single stream {s}")
    pr.gpu.sync()


def test_batched_mixed_query_counts_take_several_kernel_shapes():
    """Query counts 40, 130, 200 and 262 need four kernel shapes (one or two
    M-tiles, with or without extra rows): one launch per shape."""
    w = WORKLOADS["lingbot"]
    pr = Pair(w, seed=2, pool_pages=512)
    lengths = [12, 30, 75, 90]
    counts = [40, 130, 200, 262]
    sids = _streams(pr, lengths)
    qs = [pr.gpu_q_chunk(s, 0, [n - 1])[:c].contiguous() for s, n, c in zip(sids, lengths, counts)]
    outs = pr.gpu.attend_batched(qs, sids, 0, sm_scale=w.sm_scale)
    for s, n, c, out in zip(sids, lengths, counts, outs):
        rows = np.arange(0, c, 3)
        o, e = pr.oracle_attention(s, 0, pr.cpu_q(s, 0, [n - 1])[:c], rows=rows)
        assert_close(out[torch.from_numpy(rows).cuda()], o, e, f"stream {s} ({c} rows)")
    pr.gpu.sync()


def test_batched_32_lingbot_streams():
    """32 LingBot-shaped streams of 20 to 237 frames (most past the 71-frame
    ramp) in one call; sampled rows of every fourth stream against the oracle."""
    w = WORKLOADS["lingbot"]
    pr = Pair(w, seed=3, pool_pages=3072)
    lengths = [20 + 7 * i for i in range(32)]
    sids = _streams(pr, lengths)
    qs = [pr.gpu_q_chunk(s, 0, [n - 1]) for s, n in zip(sids, lengths)]
    outs = pr.gpu.attend_batched(qs, sids, 0, sm_scale=w.sm_scale)
    rows = np.arange(0, w.frame_tokens, 9)
    for i in range(0, 32, 4):
        s, n = sids[i], lengths[i]
        o, e = pr.oracle_attention(s, 0, pr.cpu_q(s, 0, [n - 1]), rows=rows)
        assert_close(outs[i][torch.from_numpy(rows).cuda()], o, e, f"stream {s} ({n} frames)")
    # every stream's output also agrees with its separate call
    for s, q, out in zip(sids, qs, outs):
        single = pr.gpu.attend(q, s, 0, sm_scale=w.sm_scale)
        assert float((single.float() - out.float()).abs().max()) <= 2e-2
    pr.gpu.sync()


def test_batched_errors_launch_nothing():
    from paged_kv_cache_build_gb300 import PkvError, kernel_launches
    w = WORKLOADS["tiny"]
    pr = Pair(w, layers=1)
    sids = _streams(pr, [2, 3])
    empty = pr.open()                              # nothing appended: nothing visible
    q = pr.gpu_q_chunk(sids[0], 0, [1])
    before = kernel_launches()
    with pytest.raises(PkvError) as ex:
        pr.gpu.attend_batched([q, q], [sids[0], sids[0]], 0)
    assert ex.value.code == "INVALID"
    with pytest.raises(PkvError) as ex:
        pr.gpu.attend_batched([q, q], [sids[1], empty], 0)
    assert ex.value.code == "STATE"
    with pytest.raises(PkvError) as ex:
        pr.gpu.attend_batched([q], [99], 0)
    assert kernel_launches() == before
    pr.gpu.sync()
