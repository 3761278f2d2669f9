"""fp64 softmax attention over the explicitly concatenated visible tokens
(oracle; test infrastructure only).

"LingBot-Map Paged KV Cache", sections 1-2: each new frame's tokens attend
to the keys and values of the visible pages (scale -> window -> special),
which already include the frame's own tokens; the visible table needs no
mask beyond each page's valid length. The attention is bidirectional (no
causal mask), like the "full bi-directional" DiT attention of the vLLM-Omni
architecture pages. The vLLM-Omni RFC "Reconstruction Engine", section 3.3,
is the same computation with a whole chunk's tokens as queries.

For every query row i and head h:
    s_j = sm_scale * sum_d q[i,h,d] * K[j,h,d]
    o[i,h,:] = sum_j exp(s_j - max_j s_j) V[j,h,:] / sum_j exp(s_j - max_j s_j)
over all visible tokens j. Inputs are bf16 bit patterns widened exactly to
fp64; the matrix products are library fp64 matmuls; nothing is blocked,
fused or reordered.
"""

import numpy as np


def _widen(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def gather_visible(tokens, layer, kv_lookup):
    """Concatenate the K and V rows of the visible tokens.

    tokens     provenance list (stream, frame, token) in table order, as
               returned by PagedCacheOracle.visible_tokens
    kv_lookup  callable (stream, frame, layer) -> (k, v), each bf16 bits
               [frame tokens][heads][head_dim] as given to append
    Returns (K_cat, V_cat) as bf16 bits [N][heads][head_dim].
    """
    if not tokens:
        raise ValueError("no visible tokens")
    cache = {}
    k_rows, v_rows = [], []
    for (s, f, t) in tokens:
        key = (s, f)
        if key not in cache:
            cache[key] = kv_lookup(s, f, layer)
        k, v = cache[key]
        k_rows.append(k[t])
        v_rows.append(v[t])
    return np.stack(k_rows), np.stack(v_rows)


def attend_fp64(q_bits, k_bits, v_bits, sm_scale, rows=None):
    """Softmax attention in fp64.

    q_bits [n_q][H][D], k_bits/v_bits [N][H][D] (bf16 bit patterns).
    rows: optional index array selecting the query rows to compute.
    Returns fp64 [len(rows) or n_q][H][D].
    """
    q = _widen(q_bits)
    if rows is not None:
        q = q[np.asarray(rows)]
    k = _widen(k_bits)
    v = _widen(v_bits)
    if k.shape[0] == 0:
        raise ValueError("no visible tokens")
    n_q, heads, _ = q.shape
    out = np.empty((n_q, heads, v.shape[2]), dtype=np.float64)
    for h in range(heads):
        s = sm_scale * (q[:, h, :] @ k[:, h, :].T)
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        out[:, h, :] = (p @ v[:, h, :]) / p.sum(axis=1, keepdims=True)
    return out


def frame_attend_fp64(q_bits, k_bits, v_bits, sm_scale):
    """Intra-frame attention in fp64.

    vLLM-Omni RFC "Reconstruction Engine", section 2.2: VGGT's aggregator
    alternates frame self-attention with global self-attention; section 3.3: the
    worker runs frame attention per frame before the global attention. Frame
    attention is read as the plain softmax attention of each frame's tokens over
    that frame's own tokens (bidirectional, no cache):
        out[f] = attend_fp64(q[f], k[f], v[f]) for every frame f.
    q_bits, k_bits, v_bits: bf16 bits [n_frames][tokens][H][D].
    Returns fp64 [n_frames][tokens][H][D].
    """
    q = np.asarray(q_bits, dtype=np.uint16)
    k = np.asarray(k_bits, dtype=np.uint16)
    v = np.asarray(v_bits, dtype=np.uint16)
    if q.ndim != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share the shape [n_frames][tokens][heads][head_dim]")
    out = np.empty(q.shape, dtype=np.float64)
    for f in range(q.shape[0]):
        out[f] = attend_fp64(q[f], k[f], v[f], sm_scale)
    return out


def softmax_rows_fp64(q_bits, k_bits, sm_scale, head):
    """The softmax probability rows of one head (for row-sum checks)."""
    q = _widen(q_bits)[:, head, :]
    k = _widen(k_bits)[:, head, :]
    s = sm_scale * (q @ k.T)
    s -= s.max(axis=1, keepdims=True)
    p = np.exp(s)
    return p / p.sum(axis=1, keepdims=True)
