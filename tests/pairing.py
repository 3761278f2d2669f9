"""Drive the CUDA library and the CPU oracle side by side on one call schedule.

Inputs: the GPU side gets its q/k/v from the library's own generator kernel
(pkv_synth_fill); the oracle regenerates the same values with the numpy
generator in `synth` (their bitwise equality is a test of its own). Nothing
the oracle sees comes from the GPU.
"""

import numpy as np
import torch

from oracle import PagedCacheOracle, StreamConfig, attend_fp64, gather_visible
from synth import TENSOR_K, TENSOR_Q, TENSOR_V, frame_tensor
from synth.inputs import bf16_bits_to_f64

# Required agreement of bf16 inputs with the fp64 oracle (max and mean absolute error).
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def cfg_of(w):
    from paged_kv_cache_build_gb300 import chunked_stream_cfg, frame_stream_cfg
    if w.mode == "frame":
        g = frame_stream_cfg(w.num_scale, w.window, w.n_patch, w.n_special, w.window_slots,
                             w.overlap_keyframes)
        o = StreamConfig(mode="frame", num_scale=w.num_scale, window=w.window, n_patch=w.n_patch,
                         n_special=w.n_special, window_slots=w.window_slots,
                         overlap_keyframes=w.overlap_keyframes)
    else:
        g = chunked_stream_cfg(w.chunk_size, w.sliding_window_num, w.tokens_per_frame)
        o = StreamConfig(mode="chunked", chunk_size=w.chunk_size,
                         sliding_window_num=w.sliding_window_num, tokens_per_frame=w.tokens_per_frame)
    return g, o


class Pair:
    """fp8=True pairs an FP8-page cache with the oracle: the oracle then attends
    over the keys and values as FP8 pages return them (oracle/fp8.py), and the
    pool check compares the stored codes and row exponents."""

    def __init__(self, w, seed=0, layers=None, pool_pages=None, max_streams=64, fp8=False):
        from paged_kv_cache_build_gb300 import PagedKVCache
        self.w, self.seed, self.fp8 = w, seed, fp8
        self.layers = layers or w.layers
        self.P = pool_pages or w.pool_pages
        self.gpu = PagedKVCache(self.P, w.page_size, w.heads, w.head_dim, self.layers, max_streams,
                                fp8=fp8)
        self.ora = PagedCacheOracle(self.P, w.page_size, max_streams)
        self._kv = {}
        self._kv_seen = {}

    def open(self, w=None):
        g, o = cfg_of(w or self.w)
        a = self.gpu.open_stream(g)
        b = self.ora.open_stream(o)
        assert a == b
        return a

    # ------------------------------------------------------------- inputs
    def gpu_tensor(self, sid, layer, frame, tensor, scale=1.0, n_tokens=None):
        from paged_kv_cache_build_gb300 import synth_fill
        w = self.w
        n = n_tokens or w.frame_tokens
        t = torch.empty((n, w.heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
        return synth_fill(t, self.seed, w.index, sid, layer, frame, tensor, 0, scale)

    def gpu_q_chunk(self, sid, layer, frames):
        """Queries of several frames, concatenated (a chunk's tokens)."""
        return torch.cat([self.gpu_tensor(sid, layer, f, TENSOR_Q, self.w.q_scale) for f in frames])

    def lookup(self, sid, frame, layer):
        """The K and V a frame appended (bf16 bits)."""
        key = (sid, frame, layer)
        if key not in self._kv:
            w = self.w
            self._kv[key] = (frame_tensor(self.seed, w.index, sid, layer, frame, TENSOR_K,
                                          w.frame_tokens, w.heads, w.head_dim),
                             frame_tensor(self.seed, w.index, sid, layer, frame, TENSOR_V,
                                          w.frame_tokens, w.heads, w.head_dim))
        return self._kv[key]

    def lookup_seen(self, sid, frame, layer):
        """The K and V the cache returns for that frame: as appended, or (FP8
        pages) after quantization to E4M3 codes with row exponents."""
        if not self.fp8:
            return self.lookup(sid, frame, layer)
        key = (sid, frame, layer)
        if key not in self._kv_seen:
            from oracle.fp8 import roundtrip_rows
            k, v = self.lookup(sid, frame, layer)
            self._kv_seen[key] = (roundtrip_rows(k), roundtrip_rows(v))
        return self._kv_seen[key]

    def cpu_q(self, sid, layer, frames):
        w = self.w
        return np.concatenate([frame_tensor(self.seed, w.index, sid, layer, f, TENSOR_Q,
                                            w.frame_tokens, w.heads, w.head_dim, w.q_scale)
                               for f in frames])

    # -------------------------------------------------------------- calls
    def append(self, sid, frame, layers=None):
        for layer in range(layers if layers is not None else self.layers):
            k = self.gpu_tensor(sid, layer, frame, TENSOR_K)
            v = self.gpu_tensor(sid, layer, frame, TENSOR_V)
            self.gpu.append_frame(sid, k, v, layer)
        self.ora.append_frame(sid, frame, self.w.frame_tokens)

    def rollback(self, sid):
        self.gpu.rollback_last_frame(sid)
        self.ora.rollback_last_frame(sid)

    def evict(self, sid):
        self.gpu.evict_window(sid)
        self.ora.evict_window(sid)

    # ------------------------------------------------------------- checks
    def check_meta(self, sid):
        free, idx, lens, _ = self.gpu.export_state(sid)
        assert free == self.ora.free, "free stack differs"
        o_idx, o_len = self.ora.visible_table(sid)
        assert idx == o_idx, f"page table differs: {idx} vs {o_idx}"
        assert lens == o_len, f"page lengths differ: {lens} vs {o_len}"
        assert self.gpu.visible_count(sid) == (len(o_idx), sum(o_len))

    def check_pool(self, sid, layer=0):
        """Every valid slot of every visible page holds exactly the token the
        oracle says it holds (bitwise; FP8 pages: the codes and row exponents)."""
        idx, lens = self.ora.visible_table(sid)
        if self.fp8:
            from oracle.fp8 import quantize_rows
            for p, n in zip(idx, lens):
                for kv in (0, 1):
                    codes, exps = self.gpu.read_page_fp8(p, kv, layer)
                    for slot in range(n):
                        s, f, t = self.ora.slots[p][slot]
                        want_c, want_e = quantize_rows(self.lookup(s, f, layer)[kv][t])
                        np.testing.assert_array_equal(codes[:, slot, :], want_c,
                                                      err_msg=f"page {p} slot {slot} kv {kv} codes")
                        np.testing.assert_array_equal(exps[:, slot], want_e,
                                                      err_msg=f"page {p} slot {slot} kv {kv} exponents")
            return
        for p, n in zip(idx, lens):
            for kv in (0, 1):
                page = self.gpu.read_page(p, kv, layer)
                for slot in range(n):
                    s, f, t = self.ora.slots[p][slot]
                    want = self.lookup(s, f, layer)[kv][t]
                    np.testing.assert_array_equal(page[:, slot, :], want,
                                                  err_msg=f"page {p} slot {slot} kv {kv}")

    def oracle_attention(self, sid, layer, q_bits, rows=None):
        k, v = gather_visible(self.ora.visible_tokens(sid), layer, self.lookup_seen)
        o = attend_fp64(q_bits, k, v, self.w.sm_scale, rows=rows)
        # attention-weighted mean of |v|: bounds the effect of rounding P to bf16
        e_abs_v = attend_fp64(q_bits, k, v & np.uint16(0x7FFF), self.w.sm_scale, rows=rows)
        return o, e_abs_v


def oracle_attention_all_rows(pair, sid, layer, q_bits, block=1374, workers=8):
    """Pair.oracle_attention over every query row, the rows cut into blocks that
    threads compute side by side (the oracle itself is unchanged: each block is
    one call of attend_fp64 with its `rows`)."""
    from concurrent.futures import ThreadPoolExecutor
    k, v = gather_visible(pair.ora.visible_tokens(sid), layer, pair.lookup_seen)
    v_abs = v & np.uint16(0x7FFF)
    n = q_bits.shape[0]
    blocks = [np.arange(r, min(n, r + block)) for r in range(0, n, block)]

    def one(rows):
        return (attend_fp64(q_bits, k, v, pair.w.sm_scale, rows=rows),
                attend_fp64(q_bits, k, v_abs, pair.w.sm_scale, rows=rows))

    with ThreadPoolExecutor(max_workers=workers) as ex:
        parts = list(ex.map(one, blocks))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def assert_close(gpu_out, oracle_out, e_abs_v, what=""):
    """The required max/mean tolerance, plus the bound derived from the arithmetic.
    bf16 has an 8-bit significand, so round-to-nearest is off by at most 2^-8
    relative: the output rounding contributes <= 2^-8 |o|, and rounding the
    softmax weights to bf16 before P.V (their sum stays fp32) contributes
    <= 2^-8 sum_j p_j |v_j| / sum_j p_j = 2^-8 E_p|v|. Scores are exact (bf16
    products, fp32 sums) and exp2 is within ~2^-22, hence the small slack."""
    g = bf16_bits_to_f64(gpu_out.view(torch.int16).cpu().numpy().view(np.uint16))
    err = np.abs(g - oracle_out)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    assert err.max() <= MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"
    tol = 2.0 ** -8 * (np.abs(oracle_out) + e_abs_v) + 1e-5
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond the derived bound; "
                           f"worst excess {np.max(err - tol):.3e}")
    return float(err.max()), float(err.mean())
