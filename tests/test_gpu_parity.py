"""Parity of the CUDA library with the CPU oracle (needs a GB300).

Page tables, free stacks and slot contents must match bit for bit; attention
outputs must be within the required tolerance (max abs 2e-2, mean abs 2e-3
against fp64) and within the bound derived from bf16 rounding (see
tests/pairing.py)."""

import os
import random

import numpy as np
import pytest
import torch

from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS, frame_tensor, is_keyframe, multistream_schedule
from tests.pairing import Pair, assert_close, oracle_attention_all_rows

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_build_gb300 import build
    build.build()


def test_generator_bitwise():
    from paged_kv_cache_build_gb300 import synth_fill
    cases = [(0, 1, 3, 2, 7, TENSOR_K, 262, 16, 1.0, 0), (1, 0, 0, 0, 0, TENSOR_Q, 22, 4, 1.0, 0),
             (0, 1, 31, 23, 9999, TENSOR_Q, 262, 16, 0.125, 0),
             (0, 3, 0, 0, 511, TENSOR_V, 1374, 16, 1.0, 0), (5, 4, 63, 31, 65535, TENSOR_V, 7, 32, 2.0, 100)]
    for seed, wl, s, layer, frame, tensor, n, heads, scale, tok0 in cases:
        t = torch.empty((n, heads, 64), dtype=torch.bfloat16, device="cuda")
        synth_fill(t, seed, wl, s, layer, frame, tensor, tok0, scale)
        ref = frame_tensor(seed, wl, s, layer, frame, tensor, n, heads, 64, scale, token0=tok0)
        np.testing.assert_array_equal(t.view(torch.int16).cpu().numpy().view(np.uint16), ref)
    # several frames in one launch
    t = torch.empty((3, 22, 4, 64), dtype=torch.bfloat16, device="cuda")
    synth_fill(t, 0, 0, 1, 0, 5, TENSOR_K)
    for f in range(3):
        np.testing.assert_array_equal(t[f].view(torch.int16).cpu().numpy().view(np.uint16),
                                      frame_tensor(0, 0, 1, 0, 5 + f, TENSOR_K, 22, 4, 64))


@pytest.mark.parametrize("seed", [0, 1])
def test_tiny_stream(seed):
    """Every frame: page table, free stack and slot bytes bit-exact; attention
    of all 22 query rows against the oracle."""
    w = WORKLOADS["tiny"]
    pr = Pair(w, seed)
    sid = pr.open()
    for t in range(w.frames):
        pr.append(sid, t)
        pr.check_meta(sid)
        pr.check_pool(sid)
        out = pr.gpu.attend(pr.gpu_q_chunk(sid, 0, [t]), sid, 0, sm_scale=w.sm_scale)
        o, e = pr.oracle_attention(sid, 0, pr.cpu_q(sid, 0, [t]))
        assert_close(out, o, e, f"tiny frame {t}")
        pr.evict(sid)
        pr.check_meta(sid)
    pr.gpu.sync()


def test_tiny_golden_trace_on_gpu():
    w = WORKLOADS["tiny"]
    pr = Pair(w)
    sid = pr.open()
    rows = []
    for line in open(os.path.join(GOLDEN, "tiny_trace.txt")):
        if line.startswith("#") or not line.strip():
            continue
        cols = [c.strip() for c in line.split("|")]
        rows.append([[] if c == "-" else [int(x) for x in c.split()] for c in cols])
    for t, (_, scale, window, special, sp_lens, _) in enumerate(rows):
        pr.append(sid, t)
        idx, lens, n, last = pr.gpu.build_visible_page_table(sid)
        assert idx.tolist() == scale + window + special
        assert lens.tolist() == [16] * (len(scale) + len(window)) + sp_lens
        assert n.item() == len(idx) and last.item() == sp_lens[-1]
        pr.evict(sid)


@pytest.mark.parametrize("seed", range(8))
def test_random_frame_streams(seed):
    """Random small configurations with keyframes, rollbacks and windowed resets;
    two layers so that layer > 0 appends and per-layer resets are covered."""
    rng = random.Random(seed)
    ps = rng.choice([16, 32, 64, 128, 192])
    S = rng.randint(1, 3)
    windowed = seed % 2 == 1
    w = WORKLOADS["tiny"].with_(page_size=ps, n_patch=ps, n_special=rng.randint(1, 6), num_scale=S,
                                window=rng.randint(1, 5), heads=rng.choice([1, 3, 4]),
                                window_slots=rng.randint(S + 1, 9) if windowed else 0,
                                overlap_keyframes=rng.randint(0, S) if windowed else 0)
    pr = Pair(w, seed, layers=2, pool_pages=96)
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
            assert_close(out, o, e, f"seed {seed} frame {t}")
        if is_keyframe(t, S, kf) and rng.random() > 0.15:
            pr.evict(sid)
        else:
            pr.rollback(sid)
        pr.check_meta(sid)
    pr.gpu.sync()


def test_rollback_restores_everything():
    """Section 3: append -> attend -> rollback leaves the free stack, the tables
    and the bytes of every valid slot exactly as they were."""
    w = WORKLOADS["tiny"]
    pr = Pair(w)
    sid = pr.open()
    for t in range(w.frames):
        before = pr.gpu.export_state(sid)
        pages = {p: (pr.gpu.read_page(p, 0), pr.gpu.read_page(p, 1)) for p in before[1]}
        pr.append(sid, 1000 + t)
        pr.gpu.attend(pr.gpu_q_chunk(sid, 0, [t]), sid, 0)
        pr.rollback(sid)
        after = pr.gpu.export_state(sid)
        assert after == before
        for p, n in zip(before[1], before[2]):
            np.testing.assert_array_equal(pr.gpu.read_page(p, 0)[:, :n], pages[p][0][:, :n])
            np.testing.assert_array_equal(pr.gpu.read_page(p, 1)[:, :n], pages[p][1][:, :n])
        pr.append(sid, t)
        pr.evict(sid)
    pr.gpu.sync()


def test_errors_change_nothing():
    from paged_kv_cache_build_gb300 import PkvError
    w = WORKLOADS["tiny"]
    pr = Pair(w, pool_pages=5)
    sid = pr.open()
    for t in range(3):
        pr.append(sid, t)
        pr.evict(sid)
    before = pr.gpu.export_state(sid)
    k = pr.gpu_tensor(sid, 0, 3, TENSOR_K)
    with pytest.raises(PkvError) as e:
        pr.gpu.append_frame(sid, k, k)
    assert e.value.code == "OOM"
    with pytest.raises(PkvError) as e:
        pr.gpu.rollback_last_frame(sid)
    assert e.value.code == "STATE"
    with pytest.raises(PkvError) as e:
        pr.gpu.append_frame(sid, k[:21].contiguous(), k[:21].contiguous())
    assert e.value.code == "INVALID"
    with pytest.raises(PkvError) as e:
        pr.gpu.append_frame(sid, k, k, layer=1)
    assert e.value.code == "INVALID"
    assert pr.gpu.export_state(sid) == before
    pr.gpu.sync()


def test_lingbot_stream_one_layer():
    """The 512-frame LingBot-shaped stream: tables bit-exact on every frame,
    slot bytes at the end, attention on sampled frames (all rows)."""
    w = WORKLOADS["lingbot"]
    pr = Pair(w)
    sid = pr.open()
    attend_at = {0, 7, 8, 71, 72, 300, 511}
    for t in range(w.frames):
        pr.append(sid, t)
        pr.check_meta(sid)
        q = pr.gpu_q_chunk(sid, 0, [t])
        out = pr.gpu.attend(q, sid, 0, sm_scale=w.sm_scale)
        if t in attend_at:
            o, e = pr.oracle_attention(sid, 0, pr.cpu_q(sid, 0, [t]))
            assert_close(out, o, e, f"lingbot frame {t}")
        pr.evict(sid)
    assert pr.gpu.visible_count(sid) == (71 + 13, 71 * 256 + 512 * 6)
    pr.check_pool(sid)
    pr.gpu.sync()


def test_peaked_softmax_and_odd_sizes():
    """Large-magnitude queries (a peaked softmax), n_q from 1 to a ragged 200,
    heads=1: the running-max rescaling and the row/column masking."""
    w = WORKLOADS["tiny"].with_(heads=1, q_scale=8.0)
    pr = Pair(w)
    sid = pr.open()
    for t in range(7):
        pr.append(sid, t)
        for n_q in (1, 5, 22):
            q = pr.gpu_tensor(sid, 0, t, TENSOR_Q, 8.0)[:n_q].contiguous()
            out = pr.gpu.attend(q, sid, 0, sm_scale=w.sm_scale)
            qc = frame_tensor(0, w.index, sid, 0, t, TENSOR_Q, w.frame_tokens, 1, 64, 8.0)[:n_q]
            o, e = pr.oracle_attention(sid, 0, qc)
            assert_close(out, o, e, f"peaked frame {t} n_q {n_q}")
        pr.evict(sid)
    # 200 query rows (several 64-row blocks plus a ragged tail) against 7 frames
    from paged_kv_cache_build_gb300 import synth_fill
    q = torch.empty((200, 1, 64), dtype=torch.bfloat16, device="cuda")
    synth_fill(q, 3, w.index, sid, 0, 0, TENSOR_Q, 0, 1.0)
    out = pr.gpu.attend(q, sid, 0, sm_scale=0.3)
    qc = frame_tensor(3, w.index, sid, 0, 0, TENSOR_Q, 200, 1, 64)
    from oracle import attend_fp64, gather_visible
    k, v = gather_visible(pr.ora.visible_tokens(sid), 0, pr.lookup)
    assert_close(out, attend_fp64(qc, k, v, 0.3), attend_fp64(qc, k, v & np.uint16(0x7FFF), 0.3), "200 rows")
    pr.gpu.sync()


def test_long_stream_keyframes_24_layers():
    """10,000 frames, 24 layers, keyframe interval 4: tables bit-exact on every
    frame; attention sampled every 500 frames (two layers, every 8th row)."""
    w = WORKLOADS["long"]
    frames = int(os.environ.get("PKV_LONG_FRAMES", w.frames))
    pr = Pair(w)
    sid = pr.open()
    rows = np.arange(0, w.frame_tokens, 8)
    for t in range(frames):
        pr.append(sid, t)
        if t % 10 == 0 or t > frames - 5:
            pr.check_meta(sid)
        if t % 500 == 0 or t == frames - 1:
            for layer in (t // 500 % 24, 23):
                q = pr.gpu_q_chunk(sid, layer, [t])
                out = pr.gpu.attend(q, sid, layer, sm_scale=w.sm_scale)
                o, e = pr.oracle_attention(sid, layer, pr.cpu_q(sid, layer, [t]), rows=rows)
                assert_close(out[torch.from_numpy(rows).cuda()], o, e, f"long frame {t} layer {layer}")
        if is_keyframe(t, w.num_scale, w.keyframe_interval):
            pr.evict(sid)
        else:
            pr.rollback(sid)
    pr.check_meta(sid)
    if frames == w.frames:
        kept = 8 + -(-(w.frames - 8) // 4)
        assert pr.ora.streams[sid].kept == kept == 2506
        assert len(pr.ora.streams[sid].special) == 60
    pr.check_pool(sid, layer=17)
    pr.gpu.sync()


@pytest.mark.parametrize("ps", [16, 32])
def test_extra_rows_with_small_pages(ps):
    """Chunks of 2 frames of 131 tokens, i.e. 262 queries (two M-tiles plus extra
    rows, each extra-row warp on whole tiles), on pages of 16 and 32 slots, so that
    a 64-slot tile spans four or two page blocks; 3 chunks visible, every row."""
    w = WORKLOADS["chunked"].with_(page_size=ps, chunk_size=2, tokens_per_frame=131, sliding_window_num=3,
                                   heads=2, frames=10)
    pr = Pair(w, seed=6, pool_pages=128)
    sid = pr.open()
    for c in range(5):
        frames = [2 * c, 2 * c + 1]
        for f in frames:
            pr.append(sid, f)
        pr.check_meta(sid)
        out = pr.gpu.attend_chunked(pr.gpu_q_chunk(sid, 0, frames), sid, 0, sm_scale=w.sm_scale)
        o, e = pr.oracle_attention(sid, 0, pr.cpu_q(sid, 0, frames))
        assert_close(out, o, e, f"page {ps} chunk {c}")
        pr.evict(sid)
    pr.check_pool(sid)
    pr.gpu.sync()


def test_chunked_vggt_stream():
    """RFC chunked sliding-window attention: 64 chunks of 8 x 1374 tokens, 4
    chunks visible; tables every chunk, attention of chunks 0-2 and 63 on every
    16th query row, and of chunk 3 (the first with all 4 chunks visible: 43 M-groups
    x 16 heads x 3 KV splits) on all 10,992 query rows."""
    w = WORKLOADS["chunked"]
    n_chunks = int(os.environ.get("PKV_CHUNKS", 64))
    pr = Pair(w)
    sid = pr.open()
    check = {0, 1, 2, 3, n_chunks - 1}
    for c in range(n_chunks):
        frames = list(range(c * 8, c * 8 + 8))
        for f in frames:
            pr.append(sid, f)
        pr.check_meta(sid)
        q = pr.gpu_q_chunk(sid, 0, frames)
        out = pr.gpu.attend_chunked(q, sid, 0, sm_scale=w.sm_scale)
        if c == 3:
            o, e = oracle_attention_all_rows(pr, sid, 0, pr.cpu_q(sid, 0, frames))
            assert_close(out, o, e, f"chunk {c}, all rows")
        elif c in check:
            rows = np.arange(0, q.shape[0], 16)
            o, e = pr.oracle_attention(sid, 0, pr.cpu_q(sid, 0, frames), rows=rows)
            assert_close(out[torch.from_numpy(rows).cuda()], o, e, f"chunk {c}")
        pr.evict(sid)
        pr.check_meta(sid)
    pr.check_pool(sid)
    pr.gpu.sync()


def test_multistream_shared_pool():
    """32 streams on one pool and free list, lengths 100-5000, keyframe
    intervals 1-8, windowed mode (128 slots, 8 overlap keyframes): batched
    appends (ascending ids), attends, rollbacks (descending), evicts (ascending).
    Tables and free list checked every 50 steps; attention sampled."""
    w = WORKLOADS["multistream"]
    steps_cap = int(os.environ.get("PKV_MS_STEPS", 5000))
    sched = multistream_schedule(0)
    pr = Pair(w)
    sids = [pr.open() for _ in range(w.streams)]
    assert sids == list(range(w.streams))
    n_steps = min(steps_cap, max(n for n, _ in sched))
    for g in range(n_steps):
        active = [s for s in sids if g < sched[s][0]]
        ks = [pr.gpu_tensor(s, 0, g, TENSOR_K) for s in active]
        vs = [pr.gpu_tensor(s, 0, g, TENSOR_V) for s in active]
        pr.gpu.append_frames(active, ks, vs)
        pr.ora.append_frames(active, [g] * len(active), w.frame_tokens)
        if g % 50 == 0:
            probe = active[(g // 50) % len(active)]
            out = pr.gpu.attend(pr.gpu_q_chunk(probe, 0, [g]), probe, 0, sm_scale=w.sm_scale)
            if g % 250 == 0:
                rows = np.arange(0, w.frame_tokens, 4)
                o, e = pr.oracle_attention(probe, 0, pr.cpu_q(probe, 0, [g]), rows=rows)
                assert_close(out[torch.from_numpy(rows).cuda()], o, e, f"step {g} stream {probe}")
        keep = {s for s in active if is_keyframe(g, w.num_scale, sched[s][1])}
        for s in sorted(active, reverse=True):
            if s not in keep:
                pr.rollback(s)
        for s in sorted(keep):
            pr.evict(s)
        if g % 50 == 0 or g == n_steps - 1:
            for s in active:
                pr.check_meta(s)
        for s in sids:
            if sched[s][0] == g + 1:
                pr.gpu.close_stream(s)
                pr.ora.close_stream(s)
    pr.gpu.sync()
    assert pr.gpu.free_pages() == len(pr.ora.free)
