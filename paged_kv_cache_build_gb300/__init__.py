"""Paged KV cache for streaming 3D reconstruction on GB300 (sm_103a).

The computation lives in libpkv.so (hand-written CUDA behind a C ABI, see
include/pkv.h); this package builds it and binds it with ctypes. Importing
the binding raises if the library has not been built: there is no CPU or
other fallback.
"""

from ._lib import LIB_PATH, PkvError, load  # noqa: F401


def __getattr__(name):
    # the torch-facing binding is imported lazily so that loading the library
    # (symbol checks) works without a GPU
    if name in ("PagedKVCache", "frame_stream_cfg", "chunked_stream_cfg", "synth_fill", "kernel_launches",
                "MODE_FRAME", "MODE_CHUNKED"):
        from . import cache
        return getattr(cache, name)
    raise AttributeError(name)
