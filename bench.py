#!/usr/bin/env python
"""Benchmark of the paged stream-attention cache on the LingBot-Map-shaped stream.

Workload (one "step"): a 512-frame stream, 256 patch + 6 special tokens per
frame, page_size 256, 8 scale frames, 64-frame window, special pages of
42 x 6 tokens, 16 heads x 64, bf16, every frame a keyframe. Per frame:
append (pop pages + scatter K/V), attend (visible table + paged attention of
the frame's 262 queries), evict (window page back to the free list). Each
step starts from an empty stream (pkv_stream_reset).

Metric: frame-steps/s (whole job), with attention TFLOP/s against the bf16
tensor roofline. Inputs (q, k, v for all 512 frames, 824 MB) are resident in
HBM before timing; each step reads its own 824 MB (> L2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs one independent replica per GPU (the stream does not shard; no
collective on the data path); value = frames of all ranks / max time.
"""

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "frame-steps/s and attn TFLOP/s (bf16 paged stream attn) vs GB300 roofline"
HOST_COVER_CYCLES = 400_000   # ~200 us of GPU busy-wait ahead of a per-call timing, longer than the host needs to queue the call
UNIT = "frame-steps/s"
WORKLOAD_NAME = "lingbot-1layer-512f-256p+6s-16x64-S8-W64"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--mode", choices=["graph", "eager"], default="graph")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--profile-frames", type=int, default=0,
                   help="run N frames of the stream once, eagerly, and exit (a small case for ncu)")
    p.add_argument("--profile-chunks", type=int, default=0,
                   help="run N chunks of the chunked workload once and exit (a small case for ncu)")
    p.add_argument("--profile-frame-attn", type=int, default=0,
                   help="run N intra-frame attention calls on a VGGT chunk's 8 x 1374-token frames "
                        "and exit (a small case for ncu)")
    p.add_argument("--profile-long", type=int, default=0,
                   help="run N frames of the 24-layer keyframe stream once and exit (a small case for ncu)")
    p.add_argument("--profile-append", type=int, default=0,
                   help="run N batched 32-stream appends (sources rotated over 8 sets) and exit")
    p.add_argument("--profile-batched", type=int, default=0,
                   help="N batched attention calls of 32 LingBot-shaped streams (for profiling)")
    p.add_argument("--fp8", action="store_true", help="with --profile-long: E4M3 pages")
    p.add_argument("--no-extra", action="store_true", help="skip the extra workload measurements")
    return p.parse_args()


def workload():
    from synth import WORKLOADS
    return WORKLOADS["lingbot"]


def config_dict(w):
    return {"workload": WORKLOAD_NAME, "frames_per_step": w.frames, "tokens_per_frame": w.frame_tokens,
            "heads": w.heads, "head_dim": w.head_dim, "page_size": w.page_size, "num_scale": w.num_scale,
            "window": w.window, "special_frames_per_page": w.page_size // w.n_special,
            "keyframe_interval": 1, "layers": 1, "pool_pages": w.pool_pages,
            "l2": "inputs larger than L2: each step reads 824 MB of q/k/v; the ~85 MB of visible "
                  "pages stay L2-resident across frames, as in a one-layer stream"}


def frame_flops(w, n_kv):
    return 4.0 * w.frame_tokens * n_kv * w.head_dim * w.heads


def visible_tokens(w, t):
    """Visible tokens while frame t attends (scale + window patches + specials)."""
    patch_frames = min(t + 1, w.num_scale) + min(max(t + 1 - w.num_scale, 0), w.window)
    return patch_frames * w.n_patch + (t + 1) * w.n_special


# ----------------------------------------------------------------- dist
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        if self.proc is None or not self.lines:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- peaks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def attend_traffic_per_launch(avg_visible_tokens):
    """DRAM bytes of one attention launch from the committed ncu summary, if it was
    taken on the current kernel source (else None), scaled from the captured
    frame's visible tokens to the stream's average (traffic is proportional to the
    visible K/V bytes). The capture is cold-cache (ncu flushes between passes)."""
    path = os.path.join(ROOT, "profiles", "attend_lingbot_ncu.md")
    src = os.path.join(ROOT, "paged_kv_cache_build_gb300", "csrc", "pkv_attend_tc.cu")
    if not os.path.exists(path):
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().split()[0]
    if vals.get("kernel_source_sha256_16") != digest:
        return None
    try:
        return float(vals["dram_bytes_per_launch"]) * avg_visible_tokens / float(vals["captured_visible_tokens"])
    except (KeyError, ValueError, ZeroDivisionError):
        return None


# ------------------------------------------------------------ CPU oracle
def _visible_input_lookup(w):
    """K/V of a frame for the oracle's gather, generated once. At the last frame
    only the scale and window frames' patch tokens are visible, so the other
    frames get their special tokens only (the rest is never read)."""
    import numpy as np
    from synth import TENSOR_K, TENSOR_V, frame_tensor
    last = w.frames - 1
    cache = {}

    def lookup(s, f, layer):
        if (s, f) not in cache:
            if f < w.num_scale or f > last - w.window:
                cache[(s, f)] = tuple(frame_tensor(0, w.index, s, layer, f, t, w.frame_tokens,
                                                   w.heads, 64) for t in (TENSOR_K, TENSOR_V))
            else:
                out = []
                for t in (TENSOR_K, TENSOR_V):
                    a = np.zeros((w.frame_tokens, w.heads, 64), np.uint16)
                    a[w.n_patch:] = frame_tensor(0, w.index, s, layer, f, t, w.n_special, w.heads,
                                                 64, token0=w.n_patch)
                    out.append(a)
                cache[(s, f)] = tuple(out)
        return cache[(s, f)]
    return lookup


def oracle_sample(w, seconds, rank_tag=0):
    """The CPU oracle as it stands on a bounded sample of the workload: the
    metadata state machine over the whole stream plus fp64 attention of the
    last frames (steady state, 21.5k visible tokens) until `seconds` pass."""
    from oracle import PagedCacheOracle, StreamConfig, attend_fp64, gather_visible
    from synth import TENSOR_Q, frame_tensor

    lookup = _visible_input_lookup(w)

    ora = PagedCacheOracle(w.pool_pages, w.page_size)
    sid = ora.open_stream(StreamConfig(mode="frame", num_scale=w.num_scale, window=w.window,
                                       n_patch=w.n_patch, n_special=w.n_special))
    for t in range(w.frames - 1):
        ora.append_frame(sid, t, w.frame_tokens)
        ora.evict_window(sid)
    # inputs of the sampled frames are generated before timing
    t_last = w.frames - 1
    for f in range(w.frames):
        lookup(sid, f, 0)
    q = frame_tensor(0, w.index, sid, 0, t_last, TENSOR_Q, w.frame_tokens, w.heads, 64, w.q_scale)
    ora.append_frame(sid, t_last, w.frame_tokens)
    n_frames, flops = 0, 0.0
    t0 = time.perf_counter()
    while True:
        k, v = gather_visible(ora.visible_tokens(sid), 0, lookup)
        attend_fp64(q, k, v, w.sm_scale)
        n_frames += 1
        flops += frame_flops(w, k.shape[0])
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    threads = int(os.environ.get("OMP_NUM_THREADS", cores))
    return {"value": n_frames / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "gflops_fp64": flops / el / 1e9,
            "sample": f"fp64 numpy oracle: metadata state machine over all 512 frames (untimed), then "
                      f"gather + softmax attention of steady-state frame {t_last} (21,504 visible "
                      f"tokens, 262 queries, 16 heads) repeated {n_frames}x in {el:.1f} s"}


# ------------------------------------------------------- extra workloads
def _events():
    import torch
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def extra_chunked(reps=5):
    """VGGT-style chunked attention at steady state: 4 visible chunks (43,968 slots),
    the current chunk's 10,992 queries, 16 heads x 64: attention TFLOP/s."""
    import torch
    from paged_kv_cache_build_gb300 import PagedKVCache, chunked_stream_cfg, synth_fill
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS
    w = WORKLOADS["chunked"]
    cache = PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim)
    sid = cache.open_stream(chunked_stream_cfg(w.chunk_size, w.sliding_window_num, w.tokens_per_frame))
    n_fr = w.chunk_size * w.sliding_window_num
    k = torch.empty((n_fr, w.tokens_per_frame, w.heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    synth_fill(k, 0, w.index, sid, 0, 0, TENSOR_K)
    synth_fill(v, 0, w.index, sid, 0, 0, TENSOR_V)
    for f in range(n_fr):
        cache.append_frame(sid, k[f], v[f])
        if f % w.chunk_size == w.chunk_size - 1 and f < n_fr - 1:
            cache.evict_window(sid)
    n_q = w.chunk_size * w.tokens_per_frame
    q = torch.empty((n_q, w.heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    synth_fill(q, 0, w.index, sid, 0, n_fr - w.chunk_size, TENSOR_Q, 0)
    out = torch.empty_like(q)
    for _ in range(2):
        cache.attend_chunked(q, sid, out=out, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    e0, e1 = _events()
    e0.record()
    for _ in range(reps):
        cache.attend_chunked(q, sid, out=out, sm_scale=w.sm_scale)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    n_kv = cache.visible_count(sid)[1]
    flops = 4.0 * n_q * n_kv * w.head_dim * w.heads
    cache.sync()
    cache.close()
    return {"workload": "vggt-chunked-8x1374-W4-16x64", "n_q": n_q, "visible_slots": n_kv,
            "ms_per_chunk": round(ms, 4), "attn_tflops": round(flops / (ms * 1e-3) / 1e12, 2)}


def extra_frames(reps=20, reps_small=200):
    """Intra-frame attention (pkv_attend_frames), 16 heads x 64: a VGGT chunk's 8
    frames of 1,374 tokens in one call (TFLOP/s), and one LingBot-Map frame of 262
    tokens (us per call): calls back to back from the host, and the same calls
    replayed as a CUDA graph."""
    import torch
    from paged_kv_cache_build_gb300 import PagedKVCache, synth_fill
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS
    res = {}
    for name, w, F in (("vggt_chunk", WORKLOADS["chunked"], WORKLOADS["chunked"].chunk_size),
                       ("lingbot_frame", WORKLOADS["lingbot"], 1)):
        T = w.frame_tokens
        cache = PagedKVCache(4, 16, w.heads)
        x = torch.empty((3, F, T, w.heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
        synth_fill(x[0], 0, w.index, 0, 0, 0, TENSOR_Q, 0, w.q_scale)
        synth_fill(x[1], 0, w.index, 0, 0, 0, TENSOR_K)
        synth_fill(x[2], 0, w.index, 0, 0, 0, TENSOR_V)
        out = torch.empty_like(x[0])
        n = reps if F > 1 else reps_small
        for _ in range(3):
            cache.attend_frames(x[0], x[1], x[2], out=out, sm_scale=w.sm_scale)
        torch.cuda.synchronize()
        e0, e1 = _events()
        e0.record()
        for _ in range(n):
            cache.attend_frames(x[0], x[1], x[2], out=out, sm_scale=w.sm_scale)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        flops = 4.0 * F * T * T * w.head_dim * w.heads
        # the same calls replayed as a CUDA graph: the device time without the
        # host's per-call cost (argument checks, two tensor maps, the launch)
        g = torch.cuda.CUDAGraph()
        s2 = torch.cuda.Stream()
        s2.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s2):
            with torch.cuda.graph(g, stream=s2):
                for _ in range(n):
                    cache.attend_frames(x[0], x[1], x[2], out=out, sm_scale=w.sm_scale, stream=s2)
        torch.cuda.current_stream().wait_stream(s2)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = _events()
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_dev = e0.elapsed_time(e1) / n
        res[name] = {"frames": F, "tokens": T, "us_per_call": round(ms * 1e3, 2),
                     "attn_tflops": round(flops / (ms * 1e-3) / 1e12, 2),
                     "us_per_call_graph": round(ms_dev * 1e3, 2),
                     "attn_tflops_graph": round(flops / (ms_dev * 1e-3) / 1e12, 2)}
        cache.sync()
        cache.close()
    return res


def extra_long24(frames=240, warm=100, frame_attn=False):
    """The 24-layer keyframe stream (kf 4): per frame, for each layer, append and
    attend; then evict (keyframe) or roll back. frame-steps/s over `frames` frames
    after `warm` frames (inputs from a ring of 8 frames per layer). With
    frame_attn, each layer first runs the frame's intra-frame attention
    (pkv_attend_frames), the model-shaped step of frame attention alternating
    with global attention; its q/k/v are the ring's next slot."""
    import torch
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS, is_keyframe
    w = WORKLOADS["long"]
    L, R = w.layers, 8
    cache = PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim, layers=L)
    sid = cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
    shape = (L, R, w.frame_tokens, w.heads, w.head_dim)
    k = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    v, q = torch.empty_like(k), torch.empty_like(k)
    out = torch.empty((w.frame_tokens, w.heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    for layer in range(L):
        synth_fill(k[layer], 0, w.index, sid, layer, 0, TENSOR_K)
        synth_fill(v[layer], 0, w.index, sid, layer, 0, TENSOR_V)
        synth_fill(q[layer], 0, w.index, sid, layer, 0, TENSOR_Q, 0, w.q_scale)

    out_f = torch.empty_like(out)

    def frame(t):
        for layer in range(L):
            if frame_attn:
                u = (t + 1) % R
                cache.attend_frames(q[layer, u], k[layer, u], v[layer, u], out=out_f,
                                    sm_scale=w.sm_scale)
            cache.append_frame(sid, k[layer, t % R], v[layer, t % R], layer)
            cache.attend(q[layer, t % R], sid, layer, out=out, sm_scale=w.sm_scale)
        if is_keyframe(t, w.num_scale, w.keyframe_interval):
            cache.evict_window(sid)
        else:
            cache.rollback_last_frame(sid)

    for t in range(warm):
        frame(t)
    torch.cuda.synchronize()
    e0, e1 = _events()
    e0.record()
    for t in range(warm, warm + frames):
        frame(t)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    cache.sync()
    cache.close()
    name = "model-24layer-kf4, frame + global attention" if frame_attn else "long-24layer-kf4"
    return {"workload": "%s (frames %d-%d, eager calls)" % (name, warm, warm + frames - 1),
            "frame_steps_per_s": round(frames / (ms * 1e-3), 2),
            "ms_per_frame_step": round(ms / frames, 4)}


def _percentile(xs, q):
    xs = sorted(xs)
    return xs[min(len(xs) - 1, int(round(q * (len(xs) - 1))))]


def extra_long24_full(fp8=False, frames=None, chunk=500, warm=80):
    """The 24-layer keyframe stream as configured: 10,000 frames, 256 + 6 tokens,
    16 x 64 heads, page 256, 8 scale frames, 64-frame window, keyframe interval 4
    (non-keyframes append, attend and roll back). Every frame runs through all 24
    layers from native code (pkv_stream_frames_multi: per layer append + attend,
    then evict or roll back), in calls of `chunk` frames, with a CUDA event at
    every frame boundary: frame-steps/s over the whole stream and the p50 / p99
    frame time. Inputs: a ring of 8 distinct frames per layer (the cache's pages
    and work do not depend on the values). fp8: the same on E4M3 pages."""
    import torch
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS, is_keyframe
    w = WORKLOADS["long"]
    F = frames or w.frames
    L, R = w.layers, 8
    cache = PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim, layers=L, fp8=fp8)
    sid = cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
    shape = (L, R, w.frame_tokens, w.heads, w.head_dim)
    q, k, v = (torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(3))
    out = torch.empty_like(q)
    for layer in range(L):
        synth_fill(q[layer], 0, w.index, 0, layer, 0, TENSOR_Q, 0, w.q_scale)
        synth_fill(k[layer], 0, w.index, 0, layer, 0, TENSOR_K)
        synth_fill(v[layer], 0, w.index, 0, layer, 0, TENSOR_V)
    keys = [is_keyframe(t, w.num_scale, w.keyframe_interval) for t in range(F)]
    qs, ks, vs, os_ = list(q), list(k), list(v), list(out)
    if warm:
        # warm-up on a separate stream of the same cache, then closed
        wsid = cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
        cache.stream_frames_multi(wsid, qs, ks, vs, os_, 0, warm, keys[:warm], sm_scale=w.sm_scale)
        cache.close_stream(wsid)
    torch.cuda.synchronize()
    per_frame, total_ms = [], 0.0
    for f0 in range(0, F, chunk):
        n = min(chunk, F - f0)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        cache.stream_frames_multi(sid, qs, ks, vs, os_, f0, n, keys[f0:f0 + n], sm_scale=w.sm_scale,
                                  events=ev)
        torch.cuda.synchronize()
        per_frame += [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]
        total_ms += ev[0].elapsed_time(ev[n])
    cache.sync()
    n_pages, n_kv = cache.visible_count(sid)
    cache.close()
    kf = [t for t in range(F) if keys[t]]
    return {"workload": "long-24layer-kf4, all %d frames (%s pages), native frame runs of %d"
                        % (F, "E4M3" if fp8 else "bf16", chunk),
            "frame_steps_per_s": round(F / (total_ms * 1e-3), 2),
            "ms_per_frame_step": round(total_ms / F, 4),
            "p50_ms": round(_percentile(per_frame, 0.5), 4), "p99_ms": round(_percentile(per_frame, 0.99), 4),
            "keyframe_p50_ms": round(_percentile([per_frame[t] for t in kf], 0.5), 4),
            "final_visible": {"pages": n_pages, "tokens": n_kv}}


def extra_model24(frames=1000, warm=100, chunk=500):
    """The model-shaped step, from native code (pkv_stream_model_frames): per frame,
    for each of 24 layers, the frame's intra-frame attention, then the layer's
    append and global attention over its visible pages; then evict (keyframe,
    interval 4) or roll back. The 24-layer keyframe stream's shapes; frame
    attention inputs are a second ring of 8 frames per layer. frame-steps/s and
    p50 / p99 frame time over `frames` frames after `warm` frames."""
    import torch
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS, is_keyframe
    w = WORKLOADS["long"]
    L, R = w.layers, 8
    cache = PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim, layers=L)
    sid = cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
    shape = (L, R, w.frame_tokens, w.heads, w.head_dim)
    q, k, v, fq, fk, fv = (torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(6))
    out, fout = torch.empty_like(q), torch.empty_like(q)
    for layer in range(L):
        for t, (a, b_, c_) in enumerate(((q, k, v), (fq, fk, fv))):
            synth_fill(a[layer], t, w.index, 0, layer, 0, TENSOR_Q, 0, w.q_scale)
            synth_fill(b_[layer], t, w.index, 0, layer, 0, TENSOR_K)
            synth_fill(c_[layer], t, w.index, 0, layer, 0, TENSOR_V)
    F = warm + frames
    keys = [is_keyframe(t, w.num_scale, w.keyframe_interval) for t in range(F)]
    args = [list(x) for x in (fq, fk, fv, fout, q, k, v, out)]
    cache.stream_model_frames(sid, *args, 0, warm, keys[:warm], sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    per_frame, total_ms = [], 0.0
    for f0 in range(warm, F, chunk):
        n = min(chunk, F - f0)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        cache.stream_model_frames(sid, *args, f0, n, keys[f0:f0 + n], sm_scale=w.sm_scale, events=ev)
        torch.cuda.synchronize()
        per_frame += [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]
        total_ms += ev[0].elapsed_time(ev[n])
    cache.sync()
    cache.close()
    return {"workload": "model-24layer-kf4, frame + global attention per layer (frames %d-%d, "
                        "native frame runs of %d)" % (warm, F - 1, chunk),
            "frame_steps_per_s": round(frames / (total_ms * 1e-3), 2),
            "ms_per_frame_step": round(total_ms / frames, 4),
            "p50_ms": round(_percentile(per_frame, 0.5), 4), "p99_ms": round(_percentile(per_frame, 0.99), 4)}


def extra_append(reps=20):
    """32 streams' frames appended in one batched launch (pkv_append_frames):
    2 x 262 x 16 x 64 x 2 B read and written per stream: GB/s against HBM."""
    import torch
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    from synth import TENSOR_K, TENSOR_V, WORKLOADS
    w = WORKLOADS["multistream"]
    n = w.streams
    cache = PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim, max_streams=64)
    sids = [cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
            for _ in range(n)]
    # eight source sets (8 x 68.7 MB > L2) used in turn, so every launch reads
    # its K/V from HBM
    S = 8
    kv = torch.empty((S, 2, n, w.frame_tokens, w.heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    for i in range(S):
        synth_fill(kv[i, 0], 0, w.index, 0, 0, i * n, TENSOR_K)
        synth_fill(kv[i, 1], 0, w.index, 0, 0, i * n, TENSOR_V)
    times = []
    for r in range(reps + 3):
        src = kv[r % S]
        ks, vs = [src[0, i] for i in range(n)], [src[1, i] for i in range(n)]
        e0, e1 = _events()
        torch.cuda._sleep(HOST_COVER_CYCLES)     # the host queues the call meanwhile
        e0.record()
        cache.append_frames(sids, ks, vs)
        e1.record()
        for s in sids:
            cache.evict_window(s)
        torch.cuda.synchronize()
        if r >= 3:
            times.append(e0.elapsed_time(e1))
    cache.sync()
    cache.close()
    ms = statistics.median(times)
    moved = 2.0 * 2 * n * w.frame_tokens * w.heads * w.head_dim * 2
    peaks, kind = measured_peaks()
    gbs = moved / (ms * 1e-3) / 1e9
    return {"workload": "32-stream batched append, 256+6 tokens x 16 x 64 bf16, 8 source sets "
                        "(550 MB) used in turn",
            "bytes_per_launch": int(moved), "us_per_launch": round(ms * 1e3, 2),
            "gbs": round(gbs, 1), "hbm_peak_gbs": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 3),
            "peak_source": kind}


def extra_multistream(frames=100, reps=20):
    """32 LingBot-shaped streams at steady state (`frames` frames each): one
    frame's attention for every stream, as one pkv_attend_batched call and as 32
    pkv_attend calls. frame-steps/s counts a stream's frame as one step."""
    import ctypes
    import torch
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    from paged_kv_cache_build_gb300._lib import check
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS
    w = WORKLOADS["multistream"]
    n, T, H, D = w.streams, w.frame_tokens, w.heads, w.head_dim
    cache = PagedKVCache(3072, w.page_size, H, D, max_streams=64)
    sids = [cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
            for _ in range(n)]
    R = 8
    kv = torch.empty((2, R, T, H, D), dtype=torch.bfloat16, device="cuda")
    synth_fill(kv[0], 0, w.index, 0, 0, 0, TENSOR_K)
    synth_fill(kv[1], 0, w.index, 0, 0, 0, TENSOR_V)
    for t in range(frames):
        for s in sids:
            cache.append_frame(s, kv[0, t % R], kv[1, t % R])
        if t < frames - 1:
            for s in sids:
                cache.evict_window(s)
    q = torch.empty((n * T, H, D), dtype=torch.bfloat16, device="cuda")
    synth_fill(q, 0, w.index, 0, 0, 0, TENSOR_Q, 0, w.q_scale)
    out = torch.empty_like(q)
    lib, h = cache.lib, cache.h
    c_off = (ctypes.c_int * (n + 1))(*[i * T for i in range(n + 1)])
    c_sids = (ctypes.c_int * n)(*sids)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    row = T * H * D * 2

    def batched():
        check(lib.pkv_attend_batched(h, ctypes.c_void_p(q.data_ptr()), c_off, c_sids, n, 0,
                                     ctypes.c_void_p(out.data_ptr()), ctypes.c_float(w.sm_scale),
                                     stream), h)

    def separate():
        for i, s in enumerate(sids):
            check(lib.pkv_attend(h, ctypes.c_void_p(q.data_ptr() + i * row), T, s, 0,
                                 ctypes.c_void_p(out.data_ptr() + i * row), ctypes.c_float(w.sm_scale),
                                 stream), h)

    res = {}
    for name, fn in (("batched", batched), ("separate", separate)):
        times = []
        for r in range(reps + 3):
            e0, e1 = _events()
            torch.cuda._sleep(HOST_COVER_CYCLES)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if r >= 3:
                times.append(e0.elapsed_time(e1))
        res[name] = statistics.median(times)
    n_kv = cache.visible_count(sids[0])[1]
    flops = 4.0 * T * n_kv * D * H * n
    cache.sync()
    cache.close()
    return {"workload": "32 LingBot-shaped streams x 262 queries, %d visible tokens each" % n_kv,
            "ms_batched": round(res["batched"], 4), "ms_separate": round(res["separate"], 4),
            "frame_steps_per_s_batched": round(n / (res["batched"] * 1e-3), 1),
            "frame_steps_per_s_separate": round(n / (res["separate"] * 1e-3), 1),
            "attn_tflops_batched": round(flops / (res["batched"] * 1e-3) / 1e12, 2)}


def extra_multistream_full(steps=None):
    """The multi-stream pool as configured: 32 LingBot-shaped streams on one pool
    and free list, lengths U[100, 5000] and keyframe intervals from {1, 2, 4, 8}
    (multistream_schedule(0)), windowed mode (window_size 128 KV slots, 8 overlap
    keyframes). Each global step: one batched append of every active stream
    (ascending ids), one batched attention of all of them (pkv_attend_batched),
    rollbacks of the non-keyframe streams (descending), evictions (windowed resets
    inside) of the keyframe streams (ascending); a stream closes after its last
    frame. Inputs: a ring of 4 frames per stream. frame-steps/s counts every
    stream's frame; attention TFLOP/s is over the batched attention calls."""
    import ctypes
    import torch
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    from paged_kv_cache_build_gb300._lib import check
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS, is_keyframe, multistream_schedule
    w = WORKLOADS["multistream"]
    n, T, H, D = w.streams, w.frame_tokens, w.heads, w.head_dim
    sched = multistream_schedule(0)
    n_steps = max(l for l, _ in sched) if steps is None else steps
    cache = PagedKVCache(w.pool_pages, w.page_size, H, D, max_streams=64)
    cfg = frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special, w.window_slots,
                           w.overlap_keyframes)
    sids = [cache.open_stream(cfg) for _ in range(n)]
    R = 4
    kv = torch.empty((2, R, n, T, H, D), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((R, n * T, H, D), dtype=torch.bfloat16, device="cuda")
    for r in range(R):
        synth_fill(kv[0, r], 0, w.index, 0, 0, r * n, TENSOR_K)
        synth_fill(kv[1, r], 0, w.index, 0, 0, r * n, TENSOR_V)
        synth_fill(q[r].view(n, T, H, D), 0, w.index, 0, 0, r * n, TENSOR_Q, 0, w.q_scale)
    out = torch.empty((n * T, H, D), dtype=torch.bfloat16, device="cuda")
    lib, h = cache.lib, cache.h
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    scale = ctypes.c_float(w.sm_scale)
    att_events, frames, flops = [], 0, 0.0
    torch.cuda.synchronize()
    e0, e1 = _events()
    e0.record()
    for g in range(n_steps):
        active = [s for s in sids if g < sched[s][0]]
        if not active:
            break
        r = g % R
        cache.append_frames(active, [kv[0, r, s] for s in active], [kv[1, r, s] for s in active])
        m = len(active)
        c_off = (ctypes.c_int * (m + 1))(*[i * T for i in range(m + 1)])
        c_sids = (ctypes.c_int * m)(*active)
        ea, eb = _events()
        ea.record()
        check(lib.pkv_attend_batched(h, ctypes.c_void_p(q[r].data_ptr()), c_off, c_sids, m, 0,
                                     ctypes.c_void_p(out.data_ptr()), scale, stream), h)
        eb.record()
        att_events.append((ea, eb))
        for s in active:
            flops += 4.0 * T * cache.visible_count(s)[1] * D * H
        frames += m
        keep = {s for s in active if is_keyframe(g, w.num_scale, sched[s][1])}
        for s in sorted(active, reverse=True):
            if s not in keep:
                cache.rollback_last_frame(s)
        for s in sorted(keep):
            cache.evict_window(s)
        for s in active:
            if sched[s][0] == g + 1:
                cache.close_stream(s)
    e1.record()
    torch.cuda.synchronize()
    total_ms = e0.elapsed_time(e1)
    att_ms = sum(a.elapsed_time(b) for a, b in att_events)
    cache.sync()
    cache.close()
    return {"workload": "32-stream pool, schedule 0 (lengths 100-5000, kf 1/2/4/8), windowed 128 "
                        "slots, 8 overlap keyframes, %d global steps" % len(att_events),
            "frames": frames, "frame_steps_per_s": round(frames / (total_ms * 1e-3), 1),
            "attn_ms_total": round(att_ms, 2), "attn_tflops": round(flops / (att_ms * 1e-3) / 1e12, 2),
            "ms_total": round(total_ms, 2)}


def extra_sampled(frames=150, reps=20):
    """A steady-state LingBot-shaped frame (one layer) attending to a random
    subset of its visible pages (pkv_attend_sampled): us per call at keep 1,
    1/2 and 1/4 of the pages (scale pages always kept)."""
    import torch
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS
    w = WORKLOADS["lingbot"]
    T, H, D = w.frame_tokens, w.heads, w.head_dim
    cache = PagedKVCache(w.pool_pages, w.page_size, H, D)
    sid = cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
    kv = torch.empty((2, 8, T, H, D), dtype=torch.bfloat16, device="cuda")
    synth_fill(kv[0], 0, w.index, 0, 0, 0, TENSOR_K)
    synth_fill(kv[1], 0, w.index, 0, 0, 0, TENSOR_V)
    for t in range(frames):
        cache.append_frame(sid, kv[0, t % 8], kv[1, t % 8])
        if t < frames - 1:
            cache.evict_window(sid)
    q = torch.empty((T, H, D), dtype=torch.bfloat16, device="cuda")
    synth_fill(q, 0, w.index, 0, 0, 0, TENSOR_Q, 0, w.q_scale)
    out = torch.empty_like(q)
    res = {}
    for keep in (65536, 32768, 16384):
        times = []
        for r in range(reps + 3):
            e0, e1 = _events()
            torch.cuda._sleep(HOST_COVER_CYCLES)
            e0.record()
            cache.attend_sampled(q, sid, 0, seed=r, keep=keep, out=out, sm_scale=w.sm_scale)
            e1.record()
            torch.cuda.synchronize()
            if r >= 3:
                times.append(e0.elapsed_time(e1))
        res[keep] = statistics.median(times) * 1e3
    cache.sync()
    cache.close()
    return {"workload": "lingbot frame %d, one layer, seeds 3..%d" % (frames - 1, reps + 2),
            "us_keep_all": round(res[65536], 2), "us_keep_half": round(res[32768], 2),
            "us_keep_quarter": round(res[16384], 2),
            "speedup_quarter": round(res[65536] / res[16384], 2)}


def extra_blocksparse(frames=150, reps=20):
    """A steady-state frame attending to the scale pages plus the `keep` visible
    pages of highest estimated attention mass (pkv_attend_blocksparse: the
    estimate, the selection and the attention all on the device): us per call
    keeping every page, a quarter and an eighth of the non-anchor pages. Every
    timed call follows the append of a new frame (untimed), so, as in a stream,
    the call recomputes the mean keys of the pages that frame wrote and reuses
    the cached ones of the others."""
    import torch
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS
    w = WORKLOADS["lingbot"]
    T, H, D = w.frame_tokens, w.heads, w.head_dim
    cache = PagedKVCache(w.pool_pages, w.page_size, H, D)
    sid = cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
    kv = torch.empty((2, 8, T, H, D), dtype=torch.bfloat16, device="cuda")
    synth_fill(kv[0], 0, w.index, 0, 0, 0, TENSOR_K)
    synth_fill(kv[1], 0, w.index, 0, 0, 0, TENSOR_V)
    t = 0
    for t in range(frames - 1):
        cache.append_frame(sid, kv[0, t % 8], kv[1, t % 8])
        cache.evict_window(sid)
    t = frames - 1
    q = torch.empty((T, H, D), dtype=torch.bfloat16, device="cuda")
    synth_fill(q, 0, w.index, 0, 0, 0, TENSOR_Q, 0, w.q_scale)
    out = torch.empty_like(q)
    # non-anchor pages while a frame is pending (its patch page before the eviction)
    n_other = cache.visible_count(sid)[0] - w.num_scale + 1
    res = {}
    for name, keep in (("all", n_other), ("quarter", n_other // 4), ("eighth", n_other // 8)):
        times = []
        for r in range(reps + 3):
            cache.append_frame(sid, kv[0, t % 8], kv[1, t % 8])
            t += 1
            e0, e1 = _events()
            torch.cuda._sleep(HOST_COVER_CYCLES)
            e0.record()
            cache.attend_blocksparse(q, sid, 0, keep=keep, out=out, sm_scale=w.sm_scale)
            e1.record()
            torch.cuda.synchronize()
            cache.evict_window(sid)
            if r >= 3:
                times.append(e0.elapsed_time(e1))
        res[name] = statistics.median(times) * 1e3
    cache.sync()
    cache.close()
    return {"workload": "lingbot frames %d-%d, one layer, %d non-anchor pages, a new frame before "
                        "each call" % (frames - 1, t - 1, n_other),
            "us_keep_all": round(res["all"], 2), "us_keep_quarter": round(res["quarter"], 2),
            "us_keep_eighth": round(res["eighth"], 2),
            "speedup_quarter": round(res["all"] / res["quarter"], 2)}


# ------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init(world, "nccl")

    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, kernel_launches, synth_fill
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V

    w = workload()
    F, T, H, D = w.frames, w.frame_tokens, w.heads, w.head_dim
    q = torch.empty((F, T, H, D), dtype=torch.bfloat16, device=device)
    k = torch.empty_like(q)
    v = torch.empty_like(q)
    out = torch.empty_like(q)
    synth_fill(q, 0, w.index, rank % 64, 0, 0, TENSOR_Q, 0, w.q_scale)
    synth_fill(k, 0, w.index, rank % 64, 0, 0, TENSOR_K)
    synth_fill(v, 0, w.index, rank % 64, 0, 0, TENSOR_V)

    cache = PagedKVCache(w.pool_pages, w.page_size, H, D)
    sid = cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
    lib, h = cache.lib, cache.h
    fb = T * H * D * 2
    qp = [ctypes.c_void_p(q.data_ptr() + t * fb) for t in range(F)]
    kp = [ctypes.c_void_p(k.data_ptr() + t * fb) for t in range(F)]
    vp = [ctypes.c_void_p(v.data_ptr() + t * fb) for t in range(F)]
    op = [ctypes.c_void_p(out.data_ptr() + t * fb) for t in range(F)]
    scale = ctypes.c_float(w.sm_scale)

    def check(st):
        if st != 0:
            raise RuntimeError(lib.pkv_last_error(h).decode())

    def step(stream_ptr, events=None):
        check(lib.pkv_stream_reset(h, sid, stream_ptr))
        for t in range(F):
            check(lib.pkv_append_frame(h, sid, 0, kp[t], vp[t], T, stream_ptr))
            if events is not None:
                # keep the GPU busy while the host queues the call, so that only
                # device execution lies between the two events
                torch.cuda._sleep(HOST_COVER_CYCLES)
                events[t][0].record()
            check(lib.pkv_attend(h, qp[t], T, sid, 0, op[t], scale, stream_ptr))
            if events is not None:
                events[t][1].record()
            check(lib.pkv_evict_window(h, sid, stream_ptr))

    cur = lambda: ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)  # noqa: E731
    for _ in range(max(args.warmup, 3)):
        step(cur())
    torch.cuda.synchronize()
    cache.sync()

    graph = None
    if args.mode == "graph":
        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                step(ctypes.c_void_p(s.cuda_stream))
        torch.cuda.current_stream().wait_stream(s)
        graph.replay()
        torch.cuda.synchronize()
        cache.sync()

    # ---- main timed region
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        e0.record()
        for _ in range(args.steps):
            if graph is not None:
                graph.replay()
            else:
                step(cur())
        e1.record()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(ms, world, device)
    cache.sync()

    # kernels per step, counted on one eager step (a graph replays the same launches)
    l0 = kernel_launches()
    step(cur())
    torch.cuda.synchronize()
    per_step_launches = kernel_launches() - l0
    gpu_launches = per_step_launches * args.steps

    # ---- attend launches timed with events around each call (same kernels)
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(F)]
    att_ms, att_flops, steady_ms, steady_flops = 0.0, 0.0, 0.0, 0.0
    n_att_steps = min(args.steps, 5)
    for _ in range(n_att_steps):
        step(cur(), events)
        torch.cuda.synchronize()
        for t in range(F):
            d = events[t][0].elapsed_time(events[t][1])
            fl = frame_flops(w, visible_tokens(w, t))
            att_ms += d
            att_flops += fl
            if t >= w.num_scale + w.window - 1:
                steady_ms += d
                steady_flops += fl
    cache.sync()
    attn_tflops = att_flops / (att_ms * 1e-3) / 1e12
    steady_tflops = steady_flops / (steady_ms * 1e-3) / 1e12

    # ---- end to end through the C ABI with host buffers (pinned). Each step
    # copies every frame's q, k, v from pinned host memory and every output back,
    # in chunks of 64 frames on a copy stream that runs ahead of the compute
    # stream (three H2D copies and one D2H per chunk, ordered with events), while
    # the compute stream runs each chunk's frames with one pkv_stream_frames call
    # (append, attend, evict per frame, driven from native code).
    hq, hk, hv = (torch.empty((F, T, H, D), dtype=torch.bfloat16, pin_memory=True) for _ in range(3))
    hq.copy_(q)
    hk.copy_(k)
    hv.copy_(v)
    hout = torch.empty((F, T, H, D), dtype=torch.bfloat16, pin_memory=True)
    dq, dk, dv, dout = (torch.empty((F, T, H, D), dtype=torch.bfloat16, device=device) for _ in range(4))
    chunk = 64
    copy_stream = torch.cuda.Stream(device=device)
    comp_stream = torch.cuda.current_stream(device)
    n_e2e = min(args.steps, 5)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    f0.record()
    sp = ctypes.c_void_p(comp_stream.cuda_stream)
    fbytes = T * H * D * 2                           # bytes of one [T][H][D] bf16 tensor
    for _ in range(n_e2e):
        check(lib.pkv_stream_reset(h, sid, sp))
        copy_stream.wait_stream(comp_stream)         # the previous step is done with dq/dk/dv/dout
        arrived, computed = [], []
        with torch.cuda.stream(copy_stream):
            for c0 in range(0, F, chunk):
                for dst, src in ((dq, hq), (dk, hk), (dv, hv)):
                    dst[c0:c0 + chunk].copy_(src[c0:c0 + chunk], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                arrived.append(ev)
        for ci, c0 in enumerate(range(0, F, chunk)):
            comp_stream.wait_event(arrived[ci])
            n = min(F, c0 + chunk) - c0
            off = c0 * fbytes
            check(lib.pkv_stream_frames(h, sid, 0, ctypes.c_void_p(dq.data_ptr() + off),
                                        ctypes.c_void_p(dk.data_ptr() + off),
                                        ctypes.c_void_p(dv.data_ptr() + off), n, T, None,
                                        ctypes.c_void_p(dout.data_ptr() + off), scale, sp))
            ev = torch.cuda.Event()
            ev.record(comp_stream)
            computed.append(ev)
        with torch.cuda.stream(copy_stream):
            for ci, c0 in enumerate(range(0, F, chunk)):
                copy_stream.wait_event(computed[ci])
                hout[c0:c0 + chunk].copy_(dout[c0:c0 + chunk], non_blocking=True)
        comp_stream.wait_stream(copy_stream)
    f1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    e2e_ms = max(f0.elapsed_time(f1), wall * 1e3)
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    cache.sync()
    ok = torch.equal(hout.to(device), out)   # same inputs, same kernels: identical outputs

    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    frames_total = F * args.steps * world
    value = frames_total / (ms_max * 1e-3)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "impl": "ours", "mode": args.mode,
        "config": config_dict(w),
        "attn_tflops": round(attn_tflops, 2), "attn_tflops_steady": round(steady_tflops, 2),
        "attn_us_per_frame": round(att_ms * 1e3 / (F * n_att_steps), 3),
        "roofline": {"bound": "tensor", "achieved": round(attn_tflops, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(attn_tflops / peak, 4),
                     "traffic": attend_traffic_per_launch(
                         sum(visible_tokens(w, t) for t in range(F)) / F),
                     "peak_source": f"bf16_tflops_sustained ({peak_kind}); kernel: pkv_attend call "
                                    f"(table + attention + split combine), useful flops "
                                    f"4*262*N_kv*64*16 per frame, every frame of the stream"},
        "e2e": {"value": round(F * n_e2e * world / (e2e_ms * 1e-3), 2), "unit": UNIT,
                "h2d_bytes_per_step": 3 * F * fb, "d2h_bytes_per_step": F * fb,
                "outputs_match_device_run": bool(ok)},
        "gpu_launches": int(gpu_launches),
        "launches_per_step": int(per_step_launches),
        "clocks": clocks.summary(),
    }
    if not args.no_extra and world == 1:
        # an extra that fails is reported as such; it does not cost the line
        def measured(fn, *a, **kw):
            try:
                return fn(*a, **kw)
            except Exception as exc:                    # noqa: BLE001
                return {"error": "%s: %s" % (type(exc).__name__, str(exc)[:200])}
        line["extra"] = {"chunked": measured(extra_chunked),
                         "long24_full": measured(extra_long24_full),
                         "long24_full_fp8": measured(extra_long24_full, fp8=True),
                         "multistream_full": measured(extra_multistream_full),
                         "long24": measured(extra_long24),
                         "append": measured(extra_append), "multistream": measured(extra_multistream),
                         "sampled": measured(extra_sampled), "frames": measured(extra_frames),
                         "model24": measured(extra_model24),
                         "model24_eager": measured(extra_long24, frame_attn=True),
                         "blocksparse": measured(extra_blocksparse)}
    if not args.no_cpu_baseline and world == 1:      # the host baseline: N = 1 only
        line["cpu_baseline"] = oracle_sample(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- reference arm
def run_reference(args):
    """The CPU oracle as the reference arm: each step is one steady-state frame
    of the same workload (a bounded sample), timed on the host cores."""
    world, rank, _ = dist_setup()
    if world > 1:
        dist = dist_init(world, "gloo")
        dist.barrier()
        if rank != 0:
            return
    w = workload()
    from oracle import PagedCacheOracle, StreamConfig, attend_fp64, gather_visible
    from synth import TENSOR_Q, frame_tensor

    lookup = _visible_input_lookup(w)

    ora = PagedCacheOracle(w.pool_pages, w.page_size)
    sid = ora.open_stream(StreamConfig(mode="frame", num_scale=w.num_scale, window=w.window,
                                       n_patch=w.n_patch, n_special=w.n_special))
    for t in range(w.frames - 1):
        ora.append_frame(sid, t, w.frame_tokens)
        ora.evict_window(sid)
    t_last = w.frames - 1
    for f in range(w.frames):
        lookup(sid, f, 0)
    q = frame_tensor(0, w.index, sid, 0, t_last, TENSOR_Q, w.frame_tokens, w.heads, 64, w.q_scale)

    def one():
        ora.append_frame(sid, t_last, w.frame_tokens)
        k, v = gather_visible(ora.visible_tokens(sid), 0, lookup)
        attend_fp64(q, k, v, w.sm_scale)
        ora.rollback_last_frame(sid)

    for _ in range(max(args.warmup, 1)):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    value = args.steps / el
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference", "config": config_dict(w),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "one steady-state frame (frame 511: append, gather of 21,504 "
                                       "visible tokens, fp64 attention of 262 queries x 16 heads, "
                                       "rollback) per step"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile(args):
    """N frames of the stream, eagerly, inputs for those frames only: one attend
    launch per frame, frames >= 71 in steady state (no timing, nothing printed
    but a line of counts)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_build_gb300 import PagedKVCache, frame_stream_cfg, synth_fill
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V
    w = workload()
    n = args.profile_frames
    q = torch.empty((n, w.frame_tokens, w.heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    k, v, out = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    synth_fill(q, 0, w.index, 0, 0, 0, TENSOR_Q, 0, w.q_scale)
    synth_fill(k, 0, w.index, 0, 0, 0, TENSOR_K)
    synth_fill(v, 0, w.index, 0, 0, 0, TENSOR_V)
    cache = PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim)
    sid = cache.open_stream(frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special))
    for t in range(n):
        cache.append_frame(sid, k[t], v[t])
        cache.attend(q[t], sid, out=out[t], sm_scale=w.sm_scale)
        cache.evict_window(sid)
    torch.cuda.synchronize()
    cache.sync()
    print(json.dumps({"profile_frames": n, "visible": cache.visible_count(sid)}))


def run_profile_chunked(args):
    """N chunks of the chunked workload, eagerly: one chunked attend per chunk."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_build_gb300 import PagedKVCache, chunked_stream_cfg, synth_fill
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS
    w = WORKLOADS["chunked"]
    cache = PagedKVCache(w.pool_pages, w.page_size, w.heads, w.head_dim)
    sid = cache.open_stream(chunked_stream_cfg(w.chunk_size, w.sliding_window_num, w.tokens_per_frame))
    k = torch.empty((w.chunk_size, w.tokens_per_frame, w.heads, w.head_dim), dtype=torch.bfloat16,
                    device="cuda")
    v, q = torch.empty_like(k), torch.empty_like(k)
    for c in range(args.profile_chunks):
        synth_fill(k, 0, w.index, sid, 0, c * w.chunk_size, TENSOR_K)
        synth_fill(v, 0, w.index, sid, 0, c * w.chunk_size, TENSOR_V)
        synth_fill(q, 0, w.index, sid, 0, c * w.chunk_size, TENSOR_Q)
        for f in range(w.chunk_size):
            cache.append_frame(sid, k[f], v[f])
        cache.attend_chunked(q.view(-1, w.heads, w.head_dim), sid, sm_scale=w.sm_scale)
        cache.evict_window(sid)
    torch.cuda.synchronize()
    cache.sync()
    print(json.dumps({"profile_chunks": args.profile_chunks}))


def run_profile_frame_attn(args):
    """N intra-frame attention calls (pkv_attend_frames) on one VGGT chunk's 8
    frames of 1,374 tokens, 16 heads x 64."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_build_gb300 import PagedKVCache, synth_fill
    from synth import TENSOR_K, TENSOR_Q, TENSOR_V, WORKLOADS
    w = WORKLOADS["chunked"]
    x = torch.empty((3, w.chunk_size, w.tokens_per_frame, w.heads, w.head_dim), dtype=torch.bfloat16,
                    device="cuda")
    synth_fill(x[0], 0, w.index, 0, 0, 0, TENSOR_Q)
    synth_fill(x[1], 0, w.index, 0, 0, 0, TENSOR_K)
    synth_fill(x[2], 0, w.index, 0, 0, 0, TENSOR_V)
    out = torch.empty_like(x[0])
    cache = PagedKVCache(4, 16, w.heads, w.head_dim)
    for _ in range(args.profile_frame_attn):
        cache.attend_frames(x[0], x[1], x[2], out=out, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    cache.sync()
    print(json.dumps({"profile_frame_attn": args.profile_frame_attn}))


def run_profile_long(args):
    """N frames of the 24-layer keyframe stream (bf16 or, with --fp8, E4M3 pages)
    through pkv_stream_frames_multi: 24 attention launches per frame."""
    import __graft_entry__
    __graft_entry__.build()
    extra_long24_full(fp8=args.fp8, frames=args.profile_long, chunk=args.profile_long, warm=0)
    print(json.dumps({"profile_long": args.profile_long, "fp8": args.fp8}))


def run_profile_append(args):
    """N batched appends of 32 LingBot-shaped streams, sources rotated over 8 sets."""
    import __graft_entry__
    __graft_entry__.build()
    extra_append(reps=max(args.profile_append - 3, 1))
    print(json.dumps({"profile_append": args.profile_append}))


def run_profile_batched(args):
    """N batched attention calls of 32 LingBot-shaped streams at steady state
    (then the same number of rounds of 32 separate calls)."""
    import __graft_entry__
    __graft_entry__.build()
    extra_multistream(reps=max(args.profile_batched - 3, 1))
    print(json.dumps({"profile_batched": args.profile_batched}))


def main():
    args = parse()
    if args.profile_long:
        run_profile_long(args)
    elif args.profile_batched:
        run_profile_batched(args)
    elif args.profile_append:
        run_profile_append(args)
    elif args.profile_frame_attn:
        run_profile_frame_attn(args)
    elif args.profile_chunks:
        run_profile_chunked(args)
    elif args.profile_frames:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
