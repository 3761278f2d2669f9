"""ctypes declarations of libpkv's C ABI (include/pkv.h). Marshalling only."""

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkv.so")

c_int, c_float, c_void_p, c_size_t = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
c_int32_p = ctypes.POINTER(ctypes.c_int32)

PKV_OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID", 2: "OOM", 3: "STATE", 4: "CUDA", 5: "TIMEOUT", 6: "DEVICE"}


class StreamCfg(ctypes.Structure):
    _fields_ = [("mode", c_int), ("num_scale", c_int), ("window", c_int), ("n_patch", c_int),
                ("n_special", c_int), ("window_slots", c_int), ("overlap_keyframes", c_int),
                ("chunk_size", c_int), ("sliding_window_num", c_int), ("tokens_per_frame", c_int)]


# name -> (restype, argtypes)
SIGNATURES = {
    "pkv_create": (c_int, [c_int, c_int, c_int, c_int, ctypes.POINTER(c_void_p)]),
    "pkv_create_ex": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(c_void_p)]),
    "pkv_create_fp8": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(c_void_p)]),
    "pkv_destroy": (c_int, [c_void_p]),
    "pkv_stream_open": (c_int, [c_void_p, ctypes.POINTER(StreamCfg), ctypes.POINTER(c_int)]),
    "pkv_stream_close": (c_int, [c_void_p, c_int, c_void_p]),
    "pkv_stream_reset": (c_int, [c_void_p, c_int, c_void_p]),
    "pkv_append_frame": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_int, c_void_p]),
    "pkv_append_frames": (c_int, [c_void_p, c_int, ctypes.POINTER(c_int), c_int,
                                  ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p), c_int,
                                  c_void_p]),
    "pkv_rollback_last_frame": (c_int, [c_void_p, c_int, c_void_p]),
    "pkv_evict_window": (c_int, [c_void_p, c_int, c_void_p]),
    "pkv_build_visible_page_table": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_int, c_void_p,
                                             c_void_p, c_void_p]),
    "pkv_attend": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_float, c_void_p]),
    "pkv_attend_chunked": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_float,
                                   c_void_p]),
    "pkv_attend_sampled": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_float,
                                   ctypes.c_ulonglong, c_int, c_void_p]),
    "pkv_attend_batched": (c_int, [c_void_p, c_void_p, ctypes.POINTER(c_int), ctypes.POINTER(c_int),
                                   c_int, c_int, c_void_p, c_float, c_void_p]),
    "pkv_attend_noalloc": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_float,
                                   c_void_p]),
    "pkv_attend_blocksparse": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_float,
                                       c_int, c_void_p]),
    "pkv_blocksparse_kept": (c_int, [c_void_p, ctypes.POINTER(c_int), c_int, ctypes.POINTER(c_int)]),
    "pkv_attend_frames": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_void_p,
                                  c_float, c_void_p]),
    "pkv_stream_frames": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p, c_int,
                                  c_int, c_void_p, c_void_p, c_float, c_void_p]),
    "pkv_stream_frames_multi": (c_int, [c_void_p, c_int, c_int, ctypes.POINTER(c_void_p),
                                        ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p), c_int,
                                        c_int, c_int, c_int, c_void_p, ctypes.POINTER(c_void_p),
                                        c_float, ctypes.POINTER(c_void_p), c_void_p]),
    "pkv_stream_model_frames": (c_int, [c_void_p, c_int, c_int, ctypes.POINTER(c_void_p),
                                        ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p),
                                        ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p),
                                        ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p),
                                        ctypes.POINTER(c_void_p), c_int, c_int, c_int, c_int,
                                        c_void_p, c_float, ctypes.POINTER(c_void_p), c_void_p]),
    "pkv_sync": (c_int, [c_void_p, c_void_p]),
    "pkv_visible_count": (c_int, [c_void_p, c_int, ctypes.POINTER(c_int), ctypes.POINTER(c_int)]),
    "pkv_free_pages": (c_int, [c_void_p, ctypes.POINTER(c_int)]),
    "pkv_export_state": (c_int, [c_void_p, c_int, c_int32_p, c_size_t, ctypes.POINTER(c_size_t)]),
    "pkv_read_page": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p]),
    "pkv_read_page_fp8": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]),
    "pkv_synth_fill": (c_int, [c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                               c_int, c_int, c_int, c_float, c_void_p]),
    "pkv_kernel_launches": (ctypes.c_ulonglong, []),
    "pkv_scratch_info": (c_int, [c_void_p, ctypes.POINTER(c_size_t), ctypes.POINTER(c_int)]),
    "pkv_last_error": (ctypes.c_char_p, [c_void_p]),
}

_lib = None


def load(path=LIB_PATH):
    """Load libpkv.so and declare its signatures. Raises if it is not built:
    there is no fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libpkv.so is not built ({path}); run paged_kv_cache_build_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class PkvError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status
        self.code = STATUS_NAMES.get(status, str(status))


def check(status, handle=None):
    if status != PKV_OK:
        msg = load().pkv_last_error(handle)
        raise PkvError(status, msg.decode() if msg else "")
