"""Seeded synthetic inputs for the paged stream-attention cache.

This package is shared by the tests, the CPU oracle and the benchmark. It
holds the counter-based input generator and the workload shapes only; none
of the cache's or the attention's arithmetic lives here.
"""

from .inputs import (  # noqa: F401
    TENSOR_Q, TENSOR_K, TENSOR_V, TENSOR_DRAW,
    pack_key, splitmix64, gaussian_bf16, frame_tensor, bf16_bits_to_f64,
    bf16_bits_to_f32, uniform_draw,
)
from .workloads import (  # noqa: F401
    Workload, WORKLOADS, is_keyframe, multistream_schedule,
)
