"""pkv_attend_sampled: attention over a per-layer random subset of the visible
pages (vLLM-Omni RFC section 5, AVGGT with the scale pages as anchors), against
the fp64 oracle over oracle/sampling.py's subset, and its keep-everything limit
against pkv_attend."""

import numpy as np
import pytest
import torch

from oracle import attend_fp64, gather_visible
from tests.pairing import Pair, assert_close
from synth import WORKLOADS

pytestmark = pytest.mark.gpu


def _oracle(pr, sid, layer, q_bits, seed, keep, rows=None):
    toks = pr.ora.visible_tokens_sampled(sid, seed, layer, keep)
    k, v = gather_visible(toks, layer, pr.lookup)
    o = attend_fp64(q_bits, k, v, pr.w.sm_scale, rows=rows)
    e = attend_fp64(q_bits, k, v & np.uint16(0x7FFF), pr.w.sm_scale, rows=rows)
    return o, e


def _stream(pr, frames):
    sid = pr.open()
    for t in range(frames):
        pr.append(sid, t)
        if t < frames - 1:
            pr.evict(sid)
    return sid


def test_sampled_tiny_against_oracle():
    w = WORKLOADS["tiny"]
    pr = Pair(w, seed=4, layers=2)
    sid = _stream(pr, 11)
    for layer in (0, 1):
        q = pr.gpu_q_chunk(sid, layer, [10])
        qb = pr.cpu_q(sid, layer, [10])
        for seed, keep in ((1, 0), (2, 20000), (3, 40000), (4, 65536)):
            out = pr.gpu.attend_sampled(q, sid, layer, seed=seed, keep=keep, sm_scale=w.sm_scale)
            o, e = _oracle(pr, sid, layer, qb, seed, keep)
            assert_close(out, o, e, f"layer {layer} seed {seed} keep {keep}")
    pr.gpu.sync()


def test_sampled_lingbot_two_layers():
    w = WORKLOADS["lingbot"]
    pr = Pair(w, seed=5, layers=2, pool_pages=256)
    sid = _stream(pr, 130)
    rows = np.arange(0, w.frame_tokens, 5)
    subsets = []
    for layer in (0, 1):
        q = pr.gpu_q_chunk(sid, layer, [129])
        qb = pr.cpu_q(sid, layer, [129])
        for keep in (4096, 16384):
            out = pr.gpu.attend_sampled(q, sid, layer, seed=77, keep=keep, sm_scale=w.sm_scale)
            o, e = _oracle(pr, sid, layer, qb, 77, keep, rows=rows)
            assert_close(out[torch.from_numpy(rows).cuda()], o, e, f"layer {layer} keep {keep}")
        subsets.append(pr.ora.visible_tokens_sampled(sid, 77, layer, 16384))
    assert subsets[0] != subsets[1]                 # the layers draw different subsets
    pr.gpu.sync()


def test_keep_everything_is_pkv_attend():
    w = WORKLOADS["lingbot"]
    pr = Pair(w, seed=6, pool_pages=256)
    sid = _stream(pr, 100)
    q = pr.gpu_q_chunk(sid, 0, [99])
    full = pr.gpu.attend(q, sid, 0, sm_scale=w.sm_scale)
    sampled = pr.gpu.attend_sampled(q, sid, 0, seed=123, keep=65536, sm_scale=w.sm_scale)
    assert torch.equal(full, sampled)
    pr.gpu.sync()


def test_sampled_errors():
    from paged_kv_cache_build_gb300 import PkvError, chunked_stream_cfg
    w = WORKLOADS["tiny"]
    pr = Pair(w, layers=1)
    sid = _stream(pr, 3)
    q = pr.gpu_q_chunk(sid, 0, [2])
    with pytest.raises(PkvError) as ex:
        pr.gpu.attend_sampled(q, sid, 0, keep=70000)
    assert ex.value.code == "INVALID"
    csid = pr.gpu.open_stream(chunked_stream_cfg(2, 2, w.frame_tokens))
    with pytest.raises(PkvError) as ex:
        pr.gpu.attend_sampled(q, csid, 0, keep=100)
    assert ex.value.code == "STATE"
    pr.gpu.sync()
