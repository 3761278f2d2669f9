"""Brute-force flat model of what the cache keeps, with no pages and no free list.

It pins the oracle's page machinery: after any sequence of appends,
rollbacks and evictions, the multiset of visible tokens must equal what
this model derives directly from the rules of "LingBot-Map Paged KV Cache"
(sections 2-4) and of the vLLM-Omni RFC "Reconstruction Engine" (sections
2.3 and 3.3):

frame mode   visible = patch tokens of the scale frames, patch tokens of the
             newest (at most `window`) non-scale kept frames, and the special
             tokens of every kept frame of the current window epoch. An
             eviction drops the oldest non-scale patches until window - 1
             remain; in windowed mode, once window_slots frames are kept, only
             the newest overlap_keyframes frames with live patches survive, as
             the new epoch's scale frames.
chunked mode visible = every token of the newest (at most sliding_window_num)
             chunks; an eviction keeps sliding_window_num - 1 chunks.
"""

from collections import Counter


class FlatFrameModel:
    def __init__(self, num_scale, window, n_patch, n_special, window_slots=0, overlap=0):
        self.S, self.W = num_scale, window
        self.n_patch, self.n_special = n_patch, n_special
        self.window_slots, self.overlap = window_slots, overlap
        self.frames = []   # dicts: id, scale, alive, sid

    def append(self, sid, fid):
        n_scale = sum(1 for f in self.frames if f["scale"])
        self.frames.append(dict(id=fid, sid=sid, scale=n_scale < self.S, alive=True))

    def rollback(self):
        self.frames.pop()

    def evict(self):
        live = [f for f in self.frames if not f["scale"] and f["alive"]]
        for f in live[:max(0, len(live) - (self.W - 1))]:
            f["alive"] = False
        if self.window_slots and len(self.frames) >= self.window_slots:
            survivors = [f for f in self.frames if f["alive"]][-self.overlap:] if self.overlap else []
            self.frames = [dict(f, scale=True) for f in survivors]

    def visible(self):
        c = Counter()
        for f in self.frames:
            if f["alive"]:
                for t in range(self.n_patch):
                    c[(f["sid"], f["id"], t)] += 1
            for i in range(self.n_special):
                c[(f["sid"], f["id"], self.n_patch + i)] += 1
        return c

    def patch_frames(self):
        return sum(1 for f in self.frames if f["alive"])

    def kept(self):
        return len(self.frames)


class FlatChunkModel:
    def __init__(self, sliding_window_num, tokens_per_frame):
        self.Wc, self.T = sliding_window_num, tokens_per_frame
        self.chunks = []
        self.open = False

    def append(self, sid, fid):
        if not self.open:
            self.chunks.append([])
            self.open = True
        self.chunks[-1].append((sid, fid))

    def rollback(self):
        self.chunks[-1].pop()
        if not self.chunks[-1]:
            self.chunks.pop()
            self.open = False

    def evict(self):
        self.open = False
        self.chunks = self.chunks[max(0, len(self.chunks) - (self.Wc - 1)):]

    def visible(self):
        c = Counter()
        for ch in self.chunks:
            for sid, fid in ch:
                for t in range(self.T):
                    c[(sid, fid, t)] += 1
        return c
