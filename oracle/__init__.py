"""CPU oracle for the paged stream-attention KV cache.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, obviously correct
restatement of what the cache and its attention compute: an exact integer
state machine for the page pool, the free list and the three page types, and
fp64 softmax attention over the explicitly concatenated visible tokens. It
shares no code with the CUDA library and imports nothing from it. Only the
tests, the package's smoke check and the benchmark's CPU-baseline leg may
import it; the product path never does.

Sources (page title, section):
  * "LingBot-Map Paged KV Cache: 3D reconstruction managed like LLM memory"
    (Chinese article), section 2 (paged KV cache: per-layer fixed-size pages,
    free list, scale / sliding-window / special pages, the visible page table
    in the order scale -> window -> special with last_page_len), section 3
    (keyframes: a non-keyframe is appended, attended, then rolled back) and
    section 4 (windowed inference: the cache is reset once per window of
    window_size KV slots, adjacent windows share overlap keyframes).
  * vLLM-Omni RFC "Reconstruction Engine" (issue 2727), section 2.3
    (sequence_length = sliding_window_num x chunk_size) and section 3.3
    (executor chunk loop: global attention over in-window KV plus the
    current chunk, KV append, evict the oldest chunk); section 2.2 and 3.3
    (frame attention, each frame's tokens over that frame's own tokens,
    alternating with the global attention); section 5 (KV compression: the
    per-layer random page subset of sampling.py, and the page skipping by
    estimated attention mass of blocksparse.py); section 3.4, acceleration
    dimension 5 (KV cache FP8: the E4M3 pages with power-of-two row scales of
    fp8.py).

Parity of every function here is pinned in tests/test_oracle_*.py against a
brute-force flat model, closed forms, a library softmax-attention routine and
a hand-derived page trace (tests/golden/); fp8.py against the library's
float8_e4m3fn type and the closed-form properties of its scale.
"""

from .cache import OracleError, PagedCacheOracle, StreamConfig  # noqa: F401
from .attention import attend_fp64, frame_attend_fp64, gather_visible  # noqa: F401
