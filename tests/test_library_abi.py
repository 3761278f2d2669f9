"""The C-ABI library builds for sm_103a, loads, and exports every entry point
include/pkv.h declares (no compute calls: no GPU is needed)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = []
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[\w\*\s]+?\b(pkv_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_build_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("pkv_create", "pkv_append_frame", "pkv_rollback_last_frame", "pkv_evict_window",
                     "pkv_build_visible_page_table", "pkv_attend", "pkv_attend_chunked"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_symbol(lib):
    from paged_kv_cache_build_gb300._lib import SIGNATURES
    assert set(declared_symbols()) <= set(SIGNATURES)


def test_host_side_errors_without_gpu(lib):
    """Argument checks run before any CUDA call."""
    from paged_kv_cache_build_gb300._lib import load
    L = load()
    h = ctypes.c_void_p()
    assert L.pkv_create(16, 256, 16, 128, ctypes.byref(h)) == 1      # head_dim must be 64
    assert b"head_dim" in L.pkv_last_error(None)
    assert L.pkv_create(16, 24, 16, 64, ctypes.byref(h)) == 1        # page_size
    assert L.pkv_create(0, 256, 16, 64, ctypes.byref(h)) == 1        # empty pool
    assert L.pkv_destroy(None) == 0
    assert L.pkv_synth_fill(None, 1, 1, 1, 64, 0, 0, 0, 0, 0, 0, 0, 1.0, None) == 1


def test_null_handle_is_rejected_without_gpu(lib):
    """Every entry point that takes a handle rejects a null one (PKV_ERR_INVALID)
    before any CUDA call."""
    from paged_kv_cache_build_gb300._lib import load
    L = load()
    f = ctypes.c_float(0.125)
    assert L.pkv_attend_frames(None, None, None, None, 1, 16, None, f, None) == 1
    assert b"null handle" in L.pkv_last_error(None)
    assert L.pkv_stream_frames(None, 0, 0, None, None, None, 1, 16, None, None, f, None) == 1
    assert L.pkv_attend(None, None, 1, 0, 0, None, f, None) == 1
    assert L.pkv_attend_sampled(None, None, 1, 0, 0, None, f, 1, 1, None) == 1
    assert L.pkv_evict_window(None, 0, None) == 1
    assert L.pkv_rollback_last_frame(None, 0, None) == 1


def test_every_declaration_documents_its_errors():
    """Each entry point in include/pkv.h sits under a comment that states its
    error behaviour (the two that cannot fail excepted)."""
    import re
    h = open(os.path.join(ROOT, "include", "pkv.h")).read()
    for m in re.finditer(r"\n(?:pkv_status|const char\*|unsigned long long)\s+(pkv_\w+)\(", h):
        name = m.group(1)
        before = h[:m.start()]
        end = before.rfind("*/")
        assert end > before.rfind(";"), f"{name}: no comment above the declaration"
        block = before[before.rfind("/*", 0, end):end]
        if name not in ("pkv_last_error", "pkv_kernel_launches"):
            assert "rror" in block or "Always OK" in block, f"{name}: error behaviour not stated"


def test_misaligned_generator_target_is_rejected_without_gpu(lib):
    from paged_kv_cache_build_gb300._lib import load
    L = load()
    assert L.pkv_synth_fill(ctypes.c_void_p(0x1001), 1, 1, 1, 64, 0, 0, 0, 0, 0, 0, 0, 1.0, None) == 1
    assert b"2-byte aligned" in L.pkv_last_error(None)
