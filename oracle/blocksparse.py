"""Page skipping by estimated attention mass (TEST INFRASTRUCTURE ONLY).

vLLM-Omni RFC "Reconstruction Engine", section 5 ("KV Compression Strategy
Details"): Sparse-VGGT observes that the global attention mass concentrates on a
few blocks and skips the low-weight blocks; FastVGGT keeps the initial frames
as global anchors. Read at page granularity on the LingBot-Map visible table
("LingBot-Map Paged KV Cache", section 2): a page's estimated mass is the dot
product of the frame's mean query with the page's mean key, summed over heads.
The scale pages are always kept; of the other pages, the `keep` with the
highest estimate are kept, ties going to the earlier table position, and a NaN
estimate ranks below every number. The kept pages are attended in table order.

The estimate decides which pages are kept, so it is defined to the bit, in IEEE
fp32 (the precision of the kernel that makes the same decision):
    qm[h][d] = (sum over query rows i = 0, 1, ... of q[i][h][d]) / n_q
    km[h][d] = (sum over the page's valid slots s = 0, 1, ... of K[s][h][d]) / len
    s_h      = sum over d = 0, 1, ... of (qm[h][d] * km[h][d])      (each head h)
    score    = sum over h = 0, 1, ... of s_h
every sum a running fp32 total that starts at 0, every product and quotient
rounded once (no fused multiply-add). The pages fix no order; this one (a sum per
head, then over the heads) is the reading taken because its per-head sums are
independent, so a kernel forms them at once.
"""

import math

import numpy as np


def _f32(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def pooled_mean(rows_bits):
    """fp32 mean over the first axis of bf16 bits [n][H][D], summed in order."""
    rows = _f32(rows_bits)
    acc = np.zeros(rows.shape[1:], dtype=np.float32)
    for r in rows:
        acc = np.add(acc, r, dtype=np.float32)
    return np.divide(acc, np.float32(rows.shape[0]), dtype=np.float32)


def page_score(qm, km):
    """The estimate: per head, a running fp32 sum over d in order of the fp32
    products; then a running fp32 sum of the heads' sums in head order."""
    acc = np.float32(0.0)
    H, D = qm.shape
    for h in range(H):
        s_h = np.float32(0.0)
        for d in range(D):
            s_h = np.float32(s_h + np.float32(qm[h, d] * km[h, d]))
        acc = np.float32(acc + s_h)
    return acc


def kept_positions(scores, n_anchor, keep):
    """Table positions kept, in table order: the first n_anchor, then the `keep`
    highest-scoring others (ties to the earlier position; NaN lowest)."""
    def key(e):
        s = float(scores[e])
        return -math.inf if math.isnan(s) else s
    cand = sorted(range(n_anchor, len(scores)), key=lambda e: (-key(e), e))
    chosen = set(cand[:max(keep, 0)])
    return [e for e in range(len(scores)) if e < n_anchor or e in chosen]


def page_scores(cache, sid, layer, q_bits, kv_lookup):
    """The estimate of every visible page of a frame-mode stream of the cache
    oracle, in table order. kv_lookup(stream, frame, layer) -> (k, v) bf16 bits."""
    idx, lens = cache.visible_table(sid)
    qm = pooled_mean(q_bits)
    out = []
    for p, n in zip(idx, lens):
        rows = np.stack([kv_lookup(s, f, layer)[0][t] for (s, f, t) in cache.slots[p][:n]])
        out.append(page_score(qm, pooled_mean(rows)))
    return out


def visible_tokens_blocksparse(cache, sid, layer, q_bits, keep, kv_lookup):
    """Provenance of the tokens of the kept pages, in table order."""
    idx, lens = cache.visible_table(sid)
    n_anchor = len(cache._stream(sid, "frame").scale)
    kept = kept_positions(page_scores(cache, sid, layer, q_bits, kv_lookup), n_anchor, keep)
    out = []
    for e in kept:
        out.extend(cache.slots[idx[e]][:lens[e]])
    return out
