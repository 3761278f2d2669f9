"""Python binding of libpkv: argument marshalling over the C ABI, nothing more.

Tensors are torch CUDA tensors (bf16, contiguous, [tokens][heads][64]); every
call is ordered on torch's current CUDA stream unless a stream is given. All
computation runs in the library's kernels.
"""

import ctypes

import torch

from ._lib import PkvError, StreamCfg, check, load

MODE_FRAME = 0
MODE_CHUNKED = 1


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _bf16_ptr(t, name):
    if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def frame_stream_cfg(num_scale, window, n_patch, n_special, window_slots=0, overlap_keyframes=0):
    return StreamCfg(MODE_FRAME, num_scale, window, n_patch, n_special, window_slots,
                     overlap_keyframes, 0, 0, 0)


def chunked_stream_cfg(chunk_size, sliding_window_num, tokens_per_frame):
    return StreamCfg(MODE_CHUNKED, 0, 0, 0, 0, 0, 0, chunk_size, sliding_window_num,
                     tokens_per_frame)


class PagedKVCache:
    """A page pool (per layer) with its free list, shared by up to max_streams streams."""

    def __init__(self, pool_pages, page_size, heads, head_dim=64, layers=1, max_streams=64,
                 fp8=False):
        self.lib = load()
        self.pool_pages, self.page_size, self.heads, self.head_dim = pool_pages, page_size, heads, head_dim
        self.layers = layers
        self.fp8 = bool(fp8)
        h = ctypes.c_void_p()
        create = self.lib.pkv_create_fp8 if fp8 else self.lib.pkv_create_ex
        check(create(pool_pages, page_size, heads, head_dim, layers, max_streams, ctypes.byref(h)), None)
        self.h = h

    def close(self):
        if self.h is not None and self.h.value:
            self.lib.pkv_destroy(self.h)
        self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, status):
        check(status, self.h)

    # -------------------------------------------------------------- streams
    def open_stream(self, cfg):
        sid = ctypes.c_int(-1)
        self._check(self.lib.pkv_stream_open(self.h, ctypes.byref(cfg), ctypes.byref(sid)))
        return sid.value

    def close_stream(self, sid, stream=None):
        self._check(self.lib.pkv_stream_close(self.h, sid, _stream_ptr(stream)))

    def reset_stream(self, sid, stream=None):
        self._check(self.lib.pkv_stream_reset(self.h, sid, _stream_ptr(stream)))

    def append_frame(self, sid, k, v, layer=0, stream=None):
        self._check(self.lib.pkv_append_frame(self.h, sid, layer, _bf16_ptr(k, "k"), _bf16_ptr(v, "v"),
                                              k.shape[0], _stream_ptr(stream)))

    def append_frames(self, sids, ks, vs, layer=0, stream=None):
        n = len(sids)
        ids = (ctypes.c_int * n)(*sids)
        kp = (ctypes.c_void_p * n)(*[_bf16_ptr(k, "k").value for k in ks])
        vp = (ctypes.c_void_p * n)(*[_bf16_ptr(v, "v").value for v in vs])
        self._check(self.lib.pkv_append_frames(self.h, n, ids, layer, kp, vp, ks[0].shape[0],
                                               _stream_ptr(stream)))

    def rollback_last_frame(self, sid, stream=None):
        self._check(self.lib.pkv_rollback_last_frame(self.h, sid, _stream_ptr(stream)))

    def evict_window(self, sid, stream=None):
        self._check(self.lib.pkv_evict_window(self.h, sid, _stream_ptr(stream)))

    def build_visible_page_table(self, sid, capacity=None, stream=None):
        """Returns device int32 tensors (idx[n], len[n], n[1], last_page_len[1])."""
        n_pages, _ = self.visible_count(sid)
        cap = capacity if capacity is not None else max(1, n_pages)
        dev = torch.device("cuda", torch.cuda.current_device())
        idx = torch.empty(cap, dtype=torch.int32, device=dev)
        lens = torch.empty(cap, dtype=torch.int32, device=dev)
        n = torch.empty(1, dtype=torch.int32, device=dev)
        last = torch.empty(1, dtype=torch.int32, device=dev)
        self._check(self.lib.pkv_build_visible_page_table(
            self.h, sid, ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(lens.data_ptr()), cap,
            ctypes.c_void_p(n.data_ptr()), ctypes.c_void_p(last.data_ptr()), _stream_ptr(stream)))
        return idx[:n_pages], lens[:n_pages], n, last

    def attend(self, q, sid, layer=0, out=None, sm_scale=0.0, stream=None):
        if out is None:
            out = torch.empty_like(q)
        self._check(self.lib.pkv_attend(self.h, _bf16_ptr(q, "q"), q.shape[0], sid, layer,
                                        _bf16_ptr(out, "out"), float(sm_scale), _stream_ptr(stream)))
        return out

    def attend_chunked(self, q, sid, layer=0, out=None, sm_scale=0.0, stream=None):
        if out is None:
            out = torch.empty_like(q)
        self._check(self.lib.pkv_attend_chunked(self.h, _bf16_ptr(q, "q"), q.shape[0], sid, layer,
                                                _bf16_ptr(out, "out"), float(sm_scale),
                                                _stream_ptr(stream)))
        return out

    def attend_sampled(self, q, sid, layer=0, seed=0, keep=65536, out=None, sm_scale=0.0, stream=None):
        """pkv_attend_sampled: attention over a per-layer random subset of the
        visible pages (scale pages always kept, others with probability
        keep / 65536)."""
        if out is None:
            out = torch.empty_like(q)
        self._check(self.lib.pkv_attend_sampled(self.h, _bf16_ptr(q, "q"), q.shape[0], sid, layer,
                                                _bf16_ptr(out, "out"), float(sm_scale), int(seed),
                                                int(keep), _stream_ptr(stream)))
        return out

    def attend_blocksparse(self, q, sid, layer=0, keep=0, out=None, sm_scale=0.0, stream=None):
        """pkv_attend_blocksparse: attention over the scale pages and the `keep`
        other visible pages with the highest estimated attention mass."""
        if out is None:
            out = torch.empty_like(q)
        self._check(self.lib.pkv_attend_blocksparse(self.h, _bf16_ptr(q, "q"), q.shape[0], sid,
                                                    layer, _bf16_ptr(out, "out"), float(sm_scale),
                                                    int(keep), _stream_ptr(stream)))
        return out

    def blocksparse_kept(self):
        """Table positions kept by the last attend_blocksparse call, in order."""
        buf = (ctypes.c_int * 1024)()
        n = ctypes.c_int(0)
        self._check(self.lib.pkv_blocksparse_kept(self.h, buf, 1024, ctypes.byref(n)))
        return list(buf[:n.value])

    def attend_batched(self, qs, sids, layer=0, sm_scale=0.0, stream=None):
        """pkv_attend_batched: the streams' attention in one launch. qs: one
        [n_q][heads][64] bf16 tensor per stream (packed into one buffer here);
        returns one output tensor per stream."""
        if len(qs) != len(sids):
            raise ValueError("one query tensor per stream")
        q = torch.cat([x.reshape(-1, self.heads, self.head_dim) for x in qs]).contiguous()
        out = torch.empty_like(q)
        off = [0]
        for x in qs:
            off.append(off[-1] + x.shape[0])
        n = len(sids)
        c_off = (ctypes.c_int * (n + 1))(*off)
        c_sids = (ctypes.c_int * n)(*sids)
        self._check(self.lib.pkv_attend_batched(self.h, _bf16_ptr(q, "q"), c_off, c_sids, n, layer,
                                                _bf16_ptr(out, "out"), float(sm_scale),
                                                _stream_ptr(stream)))
        return [out[off[i]:off[i + 1]] for i in range(n)]

    def attend_frames(self, q, k, v, out=None, sm_scale=0.0, stream=None):
        """pkv_attend_frames: intra-frame attention, each frame's tokens over
        that frame's own tokens. q, k, v: [n_frames][tokens][heads][64] (or one
        frame, [tokens][heads][64]) contiguous bf16 CUDA tensors."""
        if q.shape != k.shape or q.shape != v.shape:
            raise ValueError("q, k and v must have the same shape")
        if q.dim() not in (3, 4):
            raise ValueError("expected [n_frames][tokens][heads][64] or [tokens][heads][64]")
        if tuple(q.shape[-2:]) != (self.heads, self.head_dim):
            raise ValueError(f"rows must be [{self.heads}][{self.head_dim}]")
        n_frames, tokens = (1, q.shape[0]) if q.dim() == 3 else (q.shape[0], q.shape[1])
        if out is None:
            out = torch.empty_like(q)
        self._check(self.lib.pkv_attend_frames(self.h, _bf16_ptr(q, "q"), _bf16_ptr(k, "k"),
                                               _bf16_ptr(v, "v"), n_frames, tokens,
                                               _bf16_ptr(out, "out"), float(sm_scale),
                                               _stream_ptr(stream)))
        return out

    def stream_frames(self, sid, q, k, v, keyframe=None, layer=0, out=None, sm_scale=0.0,
                      stream=None):
        """pkv_stream_frames: for each frame t, append k[t]/v[t], attend q[t] into
        out[t], then evict (keyframe[t] true or keyframe None) or roll back.
        q, k, v: [n_frames][tokens][heads][64] contiguous bf16 CUDA tensors."""
        if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
            raise ValueError("q, k and v must share the shape [n_frames][tokens][heads][64]")
        n_frames, tokens = q.shape[0], q.shape[1]
        if out is None:
            out = torch.empty_like(q)
        flags = None
        if keyframe is not None:
            if len(keyframe) != n_frames:
                raise ValueError("one keyframe flag per frame")
            flags = (ctypes.c_ubyte * n_frames)(*[1 if f else 0 for f in keyframe])
        self._check(self.lib.pkv_stream_frames(self.h, sid, layer, _bf16_ptr(q, "q"),
                                               _bf16_ptr(k, "k"), _bf16_ptr(v, "v"), n_frames,
                                               tokens,
                                               ctypes.cast(flags, ctypes.c_void_p) if flags else None,
                                               _bf16_ptr(out, "out"),
                                               float(sm_scale), _stream_ptr(stream)))
        return out

    def stream_frames_multi(self, sid, qs, ks, vs, outs, frame0, n_frames, keyframe=None,
                            sm_scale=0.0, events=None, stream=None):
        """pkv_stream_frames_multi: frames frame0 .. frame0 + n_frames - 1 through
        len(qs) layers (append and attend per layer, then evict or roll back).
        qs/ks/vs/outs: one [ring][tokens][heads][64] bf16 CUDA tensor per layer;
        frame t uses slot t % ring. events: n_frames + 1 torch.cuda.Event (timing
        enabled), recorded at the frame boundaries, or None."""
        L = len(qs)
        if not (len(ks) == len(vs) == len(outs) == L):
            raise ValueError("one q, k, v and out tensor per layer")
        ring, tokens = qs[0].shape[0], qs[0].shape[1]
        arr = lambda ts, name: (ctypes.c_void_p * L)(*[_bf16_ptr(t, name).value for t in ts])  # noqa: E731
        flags = None
        if keyframe is not None:
            if len(keyframe) != n_frames:
                raise ValueError("one keyframe flag per frame")
            flags = (ctypes.c_ubyte * n_frames)(*[1 if f else 0 for f in keyframe])
        ev = None
        if events is not None:
            if len(events) != n_frames + 1:
                raise ValueError("n_frames + 1 events")
            for e in events:
                if not e.cuda_event:        # torch creates the CUDA event on its first record
                    e.record(stream)
            ev = (ctypes.c_void_p * (n_frames + 1))(*[e.cuda_event for e in events])
        self._check(self.lib.pkv_stream_frames_multi(
            self.h, sid, L, arr(qs, "q"), arr(ks, "k"), arr(vs, "v"), ring, frame0, n_frames, tokens,
            ctypes.cast(flags, ctypes.c_void_p) if flags else None, arr(outs, "out"), float(sm_scale),
            ev, _stream_ptr(stream)))

    def stream_model_frames(self, sid, fqs, fks, fvs, fouts, qs, ks, vs, outs, frame0, n_frames,
                            keyframe=None, sm_scale=0.0, events=None, stream=None):
        """pkv_stream_model_frames: as stream_frames_multi, with each layer's
        intra-frame attention (fqs/fks/fvs -> fouts, one ring per layer) before its
        append and global attention."""
        L = len(qs)
        if not all(len(x) == L for x in (ks, vs, outs, fqs, fks, fvs, fouts)):
            raise ValueError("one tensor of each kind per layer")
        ring, tokens = qs[0].shape[0], qs[0].shape[1]
        arr = lambda ts, name: (ctypes.c_void_p * L)(*[_bf16_ptr(t, name).value for t in ts])  # noqa: E731
        flags = None
        if keyframe is not None:
            if len(keyframe) != n_frames:
                raise ValueError("one keyframe flag per frame")
            flags = (ctypes.c_ubyte * n_frames)(*[1 if f else 0 for f in keyframe])
        ev = None
        if events is not None:
            if len(events) != n_frames + 1:
                raise ValueError("n_frames + 1 events")
            for e in events:
                if not e.cuda_event:        # torch creates the CUDA event on its first record
                    e.record(stream)
            ev = (ctypes.c_void_p * (n_frames + 1))(*[e.cuda_event for e in events])
        self._check(self.lib.pkv_stream_model_frames(
            self.h, sid, L, arr(fqs, "fq"), arr(fks, "fk"), arr(fvs, "fv"), arr(fouts, "fout"),
            arr(qs, "q"), arr(ks, "k"), arr(vs, "v"), arr(outs, "out"), ring, frame0, n_frames, tokens,
            ctypes.cast(flags, ctypes.c_void_p) if flags else None, float(sm_scale), ev,
            _stream_ptr(stream)))

    def attend_noalloc(self, q, sid, layer=0, out=None, sm_scale=0.0, stream=None):
        """pkv_attend_noalloc: attention whose scratch is a fixed device array."""
        if out is None:
            out = torch.empty_like(q)
        self._check(self.lib.pkv_attend_noalloc(self.h, _bf16_ptr(q, "q"), q.shape[0], sid, layer,
                                                _bf16_ptr(out, "out"), float(sm_scale),
                                                _stream_ptr(stream)))
        return out

    def sync(self, stream=None):
        self._check(self.lib.pkv_sync(self.h, _stream_ptr(stream)))

    # ---------------------------------------------------------------- state
    def visible_count(self, sid):
        n_pages, n_tokens = ctypes.c_int(), ctypes.c_int()
        self._check(self.lib.pkv_visible_count(self.h, sid, ctypes.byref(n_pages), ctypes.byref(n_tokens)))
        return n_pages.value, n_tokens.value

    def scratch_info(self):
        """(bytes, allocations) of the handle's split-KV scratch."""
        b, n = ctypes.c_size_t(), ctypes.c_int()
        self._check(self.lib.pkv_scratch_info(self.h, ctypes.byref(b), ctypes.byref(n)))
        return b.value, n.value

    def free_pages(self):
        n = ctypes.c_int()
        self._check(self.lib.pkv_free_pages(self.h, ctypes.byref(n)))
        return n.value

    def export_state(self, sid):
        """(free stack bottom..top, table idx, table len, counters) read from the device."""
        cap = self.pool_pages * 4 + 1024
        buf = (ctypes.c_int32 * cap)()
        used = ctypes.c_size_t()
        self._check(self.lib.pkv_export_state(self.h, sid, buf, cap, ctypes.byref(used)))
        w = list(buf[:used.value])
        f = w[0]
        free = w[1:1 + f]
        n = w[1 + f]
        idx = w[2 + f:2 + f + n]
        lens = w[2 + f + n:2 + f + 2 * n]
        return free, idx, lens, w[2 + f + 2 * n:]

    def read_page_fp8(self, page, kv, layer=0):
        """One page's K (kv=0) or V (kv=1) of an FP8 cache as stored: (codes uint8
        [heads][page_size][64], exponents int8 [heads][page_size])."""
        import numpy as np
        codes = np.empty((self.heads, self.page_size, self.head_dim), dtype=np.uint8)
        exps = np.empty((self.heads, self.page_size), dtype=np.int8)
        self._check(self.lib.pkv_read_page_fp8(self.h, layer, page, kv,
                                               codes.ctypes.data_as(ctypes.c_void_p),
                                               exps.ctypes.data_as(ctypes.c_void_p)))
        return codes, exps

    def read_page(self, page, kv, layer=0):
        """One page's K (kv=0) or V (kv=1) as a host uint16 array [heads][page_size][64]."""
        import numpy as np
        out = np.empty((self.heads, self.page_size, self.head_dim), dtype=np.uint16)
        self._check(self.lib.pkv_read_page(self.h, layer, page, kv, out.ctypes.data_as(ctypes.c_void_p)))
        return out


def kernel_launches():
    """Kernels libpkv has launched in this process."""
    return int(load().pkv_kernel_launches())


def synth_fill(out, seed, workload, stream_id, layer, frame0, tensor, token0=0, scale=1.0, stream=None):
    """Fill a device bf16 tensor [n_frames][n_tokens][heads][head_dim] (or
    [n_tokens][heads][head_dim] for one frame) with the counter-based inputs."""
    lib = load()
    shape = out.shape if out.dim() == 4 else (1,) + tuple(out.shape)
    n_frames, n_tokens, heads, head_dim = shape
    check(lib.pkv_synth_fill(_bf16_ptr(out, "out"), n_frames, n_tokens, heads, head_dim, seed, workload,
                             stream_id, layer, frame0, tensor, token0, float(scale), _stream_ptr(stream)))
    return out


__all__ = ["PagedKVCache", "PkvError", "frame_stream_cfg", "chunked_stream_cfg", "synth_fill",
           "kernel_launches",
           "MODE_FRAME", "MODE_CHUNKED"]
