"""Exact state machine of the paged KV cache (oracle; test infrastructure only).

The pool holds `pool_pages` pages of `page_size` token slots (per layer; the
layers share one page table, so the state machine is layer-free). Instead of
bytes, every valid slot records where its token came from: the tuple
(stream id, frame id, token index inside the frame). Token values are looked
up from the caller's inputs only when attention is computed, so the state
here is exactly "which token sits in which slot of which page".

Frame mode follows "LingBot-Map Paged KV Cache", section 2:
  * one frame's n_patch patch tokens fill exactly one page (n_patch ==
    page_size); the first num_scale frames' pages are scale pages and are
    never evicted; later frames' pages enter the sliding window;
  * pages of frames that leave the window go straight back to the free list,
    where the next frame reuses them;
  * every frame's n_special special tokens are appended to special pages,
    floor(page_size / n_special) frames per page (42 x 6 = 252 of 256 slots),
    and special pages are never recycled;
  * the visible table lists scale pages, then window pages (oldest first),
    then special pages in allocation order; the last page's fill is
    last_page_len.
Section 3: a non-keyframe is appended, attended and rolled back; the caller
decides which frames are keyframes. Section 4: in windowed mode a window
holds window_slots KV slots (one slot = one cached keyframe); when it is
full the cache is reset and the last overlap_keyframes keyframes carry over.

Chunked mode follows the vLLM-Omni RFC "Reconstruction Engine", sections 2.3
and 3.3: frames are grouped into chunks of chunk_size frames whose tokens
are packed into the chunk's own pages; attention covers the most recent
sliding_window_num chunks including the current one; after a chunk's
attention the oldest chunks are evicted so that sliding_window_num - 1 stay.

Readings where the pages are silent (each is stated in the design notes):
  * the free list is a LIFO stack that initially pops pages 0, 1, 2, ...;
  * append pops the patch page first, then (if needed) a new special page;
    rollback pushes them back in the reverse order, restoring the stack;
  * the window at attention time holds at most `window` pages including
    the current frame's; eviction runs after attention and trims the window
    to window - 1 pages;
  * special pages hold floor(page_size / n_special) frames each; a new one is
    opened when the current one is full;
  * windowed reset happens inside eviction, as soon as the cache holds
    window_slots cached keyframes. The last overlap_keyframes held patch
    pages become the new window's scale pages (their KV stays in place);
    their special tokens are copied, in order, into freshly popped special
    pages (popped before anything is freed); then the other held patch pages
    (scale pages, then window pages oldest first) and the old special pages
    (in order) are pushed on the free stack;
  * closing a stream pushes its held patch pages (scale, then window oldest
    first) and then its special pages (in order); chunked streams push their
    chunks' pages oldest chunk first, in page order.
"""

from dataclasses import dataclass


class OracleError(Exception):
    """Raised with code INVALID, OOM or STATE; the state is left unchanged."""

    def __init__(self, code, msg):
        super().__init__(f"{code}: {msg}")
        self.code = code


@dataclass(frozen=True)
class StreamConfig:
    mode: str = "frame"            # "frame" or "chunked"
    num_scale: int = 0
    window: int = 0
    n_patch: int = 0
    n_special: int = 0
    window_slots: int = 0          # 0: not windowed
    overlap_keyframes: int = 0
    chunk_size: int = 0
    sliding_window_num: int = 0
    tokens_per_frame: int = 0


class _FrameStream:
    def __init__(self, cfg, page_size):
        self.cfg = cfg
        self.f_sp = page_size // cfg.n_special
        self.scale = []       # [(page, frame_id, kept_index)]
        self.window = []      # [(page, frame_id, kept_index)], oldest first
        self.special = []     # pages in allocation order
        self.sp_len = 0       # filled slots of the last special page
        self.kept = 0         # cached keyframes (KV slots) in this window
        self.undo = None


class _Chunk:
    def __init__(self):
        self.pages = []
        self.length = 0       # tokens
        self.frames = 0


class _ChunkStream:
    def __init__(self, cfg):
        self.cfg = cfg
        self.chunks = []      # oldest first
        self.open = False     # the newest chunk still takes frames
        self.undo = None


class PagedCacheOracle:
    def __init__(self, pool_pages, page_size, max_streams=64):
        if pool_pages < 1 or page_size < 1:
            raise OracleError("INVALID", "empty pool")
        self.P = pool_pages
        self.page_size = page_size
        self.max_streams = max_streams
        # Free stack: the top is the end of the list, so pops return 0, 1, 2, ...
        self.free = [pool_pages - 1 - i for i in range(pool_pages)]
        self.slots = {}       # page -> list of page_size provenance entries (or None)
        self.streams = {}

    # ----------------------------------------------------------------- pool
    def _pop(self):
        p = self.free.pop()
        self.slots[p] = [None] * self.page_size
        return p

    def _push(self, p):
        self.free.append(p)
        self.slots.pop(p, None)

    def free_count(self):
        return len(self.free)

    # -------------------------------------------------------------- streams
    def open_stream(self, cfg):
        if cfg.mode == "frame":
            if cfg.n_patch != self.page_size or cfg.n_special < 1 or cfg.n_special > self.page_size:
                raise OracleError("INVALID", "frame mode needs n_patch == page_size, 1 <= n_special <= page_size")
            if cfg.num_scale < 0 or cfg.window < 1:
                raise OracleError("INVALID", "window must be >= 1")
            if cfg.window_slots and not (0 <= cfg.overlap_keyframes <= cfg.num_scale
                                         and cfg.overlap_keyframes < cfg.window_slots):
                raise OracleError("INVALID", "overlap_keyframes must be <= num_scale and < window_slots")
        elif cfg.mode == "chunked":
            if cfg.chunk_size < 1 or cfg.sliding_window_num < 1 or cfg.tokens_per_frame < 1:
                raise OracleError("INVALID", "chunked mode needs positive chunk_size, window, tokens")
        else:
            raise OracleError("INVALID", "unknown mode")
        for sid in range(self.max_streams):
            if sid not in self.streams:
                self.streams[sid] = (_FrameStream(cfg, self.page_size) if cfg.mode == "frame"
                                     else _ChunkStream(cfg))
                return sid
        raise OracleError("OOM", "no free stream id")

    def _stream(self, sid, mode=None):
        st = self.streams.get(sid)
        if st is None:
            raise OracleError("INVALID", f"stream {sid} is not open")
        if mode is not None and st.cfg.mode != mode:
            raise OracleError("STATE", f"stream {sid} is not in {mode} mode")
        return st

    def close_stream(self, sid):
        st = self._stream(sid)
        if st.cfg.mode == "frame":
            for p, _, _ in st.scale + st.window:
                self._push(p)
            for p in st.special:
                self._push(p)
        else:
            for c in st.chunks:
                for p in c.pages:
                    self._push(p)
        del self.streams[sid]

    # ----------------------------------------------------------- frame mode
    def _append_plan(self, st):
        """Validate one frame-mode append; return (to_scale, new_special)."""
        cfg = st.cfg
        to_scale = len(st.scale) < cfg.num_scale
        if not to_scale and len(st.window) == cfg.window:
            raise OracleError("STATE", "window is full: evict before appending")
        new_sp = (not st.special) or (st.sp_len + cfg.n_special > st.f_sp * cfg.n_special)
        return to_scale, new_sp

    def append_frame(self, sid, frame_id, n_tokens):
        st = self._stream(sid)
        if st.cfg.mode == "chunked":
            return self._append_chunked(sid, st, frame_id, n_tokens)
        cfg = st.cfg
        if n_tokens != cfg.n_patch + cfg.n_special:
            raise OracleError("INVALID", "n_tokens must be n_patch + n_special")
        to_scale, new_sp = self._append_plan(st)
        if len(self.free) < 1 + new_sp:
            raise OracleError("OOM", "free list exhausted")
        self._do_append(sid, st, frame_id, to_scale, new_sp)

    def _do_append(self, sid, st, frame_id, to_scale, new_sp):
        cfg = st.cfg
        page = self._pop()
        for t in range(cfg.n_patch):
            self.slots[page][t] = (sid, frame_id, t)
        (st.scale if to_scale else st.window).append((page, frame_id, st.kept))
        sp_before = st.sp_len
        if new_sp:
            st.special.append(self._pop())
            st.sp_len = 0
        sp_page = st.special[-1]
        for i in range(cfg.n_special):
            self.slots[sp_page][st.sp_len + i] = (sid, frame_id, cfg.n_patch + i)
        st.sp_len += cfg.n_special
        st.kept += 1
        st.undo = dict(page=page, to_scale=to_scale, new_sp=new_sp, sp_before=sp_before)

    def append_frames(self, sids, frame_ids, n_tokens):
        """Several frame-mode streams' appends, in the order given. Validated as a
        whole (pages needed against the free count) before any of them runs."""
        if len(set(sids)) != len(sids):
            raise OracleError("INVALID", "a stream appears twice in one batch")
        need = 0
        for sid in sids:
            st = self._stream(sid, "frame")
            if n_tokens != st.cfg.n_patch + st.cfg.n_special:
                raise OracleError("INVALID", "n_tokens must be n_patch + n_special")
            need += 1 + self._append_plan(st)[1]
        if len(self.free) < need:
            raise OracleError("OOM", "free list exhausted")
        for sid, fid in zip(sids, frame_ids):
            st = self.streams[sid]
            self._do_append(sid, st, fid, *self._append_plan(st))

    def rollback_last_frame(self, sid):
        st = self._stream(sid)
        if st.undo is None:
            raise OracleError("STATE", "nothing to roll back")
        if st.cfg.mode == "chunked":
            return self._rollback_chunked(st)
        u, cfg = st.undo, st.cfg
        if u["new_sp"]:
            self._push(st.special.pop())
        else:
            sp_page = st.special[-1]
            for i in range(st.sp_len - cfg.n_special, st.sp_len):
                self.slots[sp_page][i] = None
        st.sp_len = u["sp_before"]
        page, _, _ = (st.scale if u["to_scale"] else st.window).pop()
        assert page == u["page"]
        self._push(page)
        st.kept -= 1
        st.undo = None

    def evict_window(self, sid):
        st = self._stream(sid)
        if st.cfg.mode == "chunked":
            return self._evict_chunked(st)
        cfg = st.cfg
        n_evict = max(0, len(st.window) - (cfg.window - 1))
        reset = cfg.window_slots > 0 and st.kept >= cfg.window_slots
        if reset:
            held = len(st.scale) + len(st.window) - n_evict
            carried = min(cfg.overlap_keyframes, held)
            n_new = -(-carried // st.f_sp)
            if len(self.free) + n_evict < n_new:
                raise OracleError("OOM", "free list exhausted by the window reset")
        for _ in range(n_evict):
            page, _, _ = st.window.pop(0)
            self._push(page)
        st.undo = None
        if reset:
            self._reset_window(st)

    def _reset_window(self, st):
        cfg = st.cfg
        held = st.scale + st.window
        carried = held[len(held) - min(cfg.overlap_keyframes, len(held)):]
        n_new = -(-len(carried) // st.f_sp)
        new_special = [self._pop() for _ in range(n_new)]
        for i, (_, _, kept_index) in enumerate(carried):
            src = self.slots[st.special[kept_index // st.f_sp]]
            dst = self.slots[new_special[i // st.f_sp]]
            s0 = (kept_index % st.f_sp) * cfg.n_special
            d0 = (i % st.f_sp) * cfg.n_special
            dst[d0:d0 + cfg.n_special] = src[s0:s0 + cfg.n_special]
        carried_pages = {p for p, _, _ in carried}
        for p, _, _ in held:
            if p not in carried_pages:
                self._push(p)
        for p in st.special:
            self._push(p)
        st.scale = [(p, fid, i) for i, (p, fid, _) in enumerate(carried)]
        st.window = []
        st.special = new_special
        st.sp_len = (len(carried) - (n_new - 1) * st.f_sp) * cfg.n_special if n_new else 0
        st.kept = len(carried)

    # --------------------------------------------------------- chunked mode
    def _append_chunked(self, sid, st, frame_id, n_tokens):
        cfg, ps = st.cfg, self.page_size
        if n_tokens != cfg.tokens_per_frame:
            raise OracleError("INVALID", "n_tokens must be tokens_per_frame")
        new_chunk = not st.open
        if new_chunk and len(st.chunks) == cfg.sliding_window_num:
            raise OracleError("STATE", "window holds sliding_window_num chunks: evict first")
        if not new_chunk and st.chunks[-1].frames == cfg.chunk_size:
            raise OracleError("STATE", "chunk is full: evict before the next chunk")
        length = 0 if new_chunk else st.chunks[-1].length
        have = 0 if new_chunk else len(st.chunks[-1].pages)
        need = -(-(length + n_tokens) // ps) - have
        if len(self.free) < need:
            raise OracleError("OOM", "free list exhausted")
        if new_chunk:
            st.chunks.append(_Chunk())
            st.open = True
        c = st.chunks[-1]
        for _ in range(need):
            c.pages.append(self._pop())
        for t in range(n_tokens):
            pos = c.length + t
            self.slots[c.pages[pos // ps]][pos % ps] = (sid, frame_id, t)
        c.length += n_tokens
        c.frames += 1
        st.undo = dict(n_new=need, new_chunk=new_chunk, n_tokens=n_tokens)

    def _rollback_chunked(self, st):
        u, ps = st.undo, self.page_size
        c = st.chunks[-1]
        for pos in range(c.length - u["n_tokens"], c.length):
            page = c.pages[pos // ps]
            if page in self.slots:
                self.slots[page][pos % ps] = None
        c.length -= u["n_tokens"]
        c.frames -= 1
        for _ in range(u["n_new"]):
            self._push(c.pages.pop())
        if u["new_chunk"]:
            st.chunks.pop()
            st.open = False
        st.undo = None

    def _evict_chunked(self, st):
        st.open = False
        while len(st.chunks) > st.cfg.sliding_window_num - 1:
            for p in st.chunks.pop(0).pages:
                self._push(p)
        st.undo = None

    def current_chunk_tokens(self, sid):
        st = self._stream(sid, "chunked")
        return st.chunks[-1].length if st.open else 0

    # ---------------------------------------------------------------- table
    def visible_table(self, sid):
        """(page ids, valid lengths) in attention order; last_page_len is lens[-1]."""
        st = self._stream(sid)
        if st.cfg.mode == "chunked":
            idx, lens = [], []
            for c in st.chunks:
                for k, p in enumerate(c.pages):
                    idx.append(p)
                    lens.append(min(self.page_size, c.length - k * self.page_size))
            return idx, lens
        cfg = st.cfg
        idx = [p for p, _, _ in st.scale] + [p for p, _, _ in st.window] + list(st.special)
        lens = [self.page_size] * (len(st.scale) + len(st.window))
        if st.special:
            lens += [st.f_sp * cfg.n_special] * (len(st.special) - 1) + [st.sp_len]
        return idx, lens

    def visible_tokens(self, sid):
        """Provenance of every visible token, in table order."""
        idx, lens = self.visible_table(sid)
        out = []
        for p, n in zip(idx, lens):
            out.extend(self.slots[p][:n])
        return out

    def visible_tokens_sampled(self, sid, seed, layer, keep):
        """Provenance of the visible tokens of the pages a layer keeps under the
        per-layer random subset (oracle/sampling.py): frame mode, scale pages
        always kept."""
        from .sampling import kept_positions
        st = self._stream(sid, "frame")
        idx, lens = self.visible_table(sid)
        out = []
        for e in kept_positions(len(idx), len(st.scale), seed, layer, keep):
            out.extend(self.slots[idx[e]][:lens[e]])
        return out

    def snapshot(self, sid=None):
        """Metadata and the provenance of every valid slot, for identity checks."""
        snap = {"free": list(self.free), "streams": {}}
        for s, st in self.streams.items():
            if sid is not None and s != sid:
                continue
            if st.cfg.mode == "frame":
                meta = (tuple(st.scale), tuple(st.window), tuple(st.special), st.sp_len, st.kept)
            else:
                meta = (tuple((tuple(c.pages), c.length, c.frames) for c in st.chunks), st.open)
            snap["streams"][s] = (meta, tuple(self.visible_table(s)[0]),
                                  tuple(self.visible_tokens(s)))
        return snap

    def patch_pages_in_use(self, sid):
        st = self._stream(sid, "frame")
        return len(st.scale) + len(st.window)
