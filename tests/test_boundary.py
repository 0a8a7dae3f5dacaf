"""The C-ABI library builds, loads and exports exactly what include/pa.h
declares; host-side validation answers without touching a GPU."""
import ctypes as C
import os
import re
import subprocess

import pytest

import paged_kv_cache_gb300 as pa
from paged_kv_cache_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text))


@pytest.fixture(scope="module")
def lib():
    path = B.build()
    return pa.load_library(path)


def test_exports_match_header(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == declared_functions()
    assert set(pa.EXPORTED) == declared_functions()
    for name in declared_functions():
        assert hasattr(lib, name)


def test_library_is_sm103a_and_self_contained(lib):
    out = subprocess.run(["ldd", B.LIB], capture_output=True, text=True).stdout
    assert "libcudart" not in out  # runtime linked statically
    assert "libcuda.so" not in out  # driver entry points resolved at run time


def test_page_bytes_and_workspace(lib):
    g = pa.geom(32, 8, 64, 16, 2, 128, 65536)
    assert pa.pa_page_bytes(g) == 32768
    assert pa.pa_page_bytes(pa.geom(8, 2, 64, 1, 1, 4, 16)) == 8192
    assert pa.pa_page_bytes(pa.geom(16, 4, 128, 1, 4, 512, 65536)) == 32768
    assert pa.pa_page_bytes(pa.geom(32, 7, 64, 1, 1, 1, 1)) == 0  # Hq not a multiple of Hkv
    w1 = pa.pa_decode_workspace_size(g, 64, 2048)
    w2 = pa.pa_decode_workspace_size(g, 256, 16384)
    assert 0 < w1 < w2
    assert w1 % 256 == 0
    assert pa.pa_decode_workspace_size(g, -1, 10) == 0


def test_status_strings(lib):
    for code in range(6):
        s = pa.pa_status_string(code)
        assert s.startswith("PA_")
    assert "unknown" in pa.pa_status_string(99)


def test_validation_without_gpu(lib):
    g = pa.geom(8, 2, 64, 1, 1, 4, 8)
    NULL = None
    # null geometry, bad layer, negative sizes: rejected before any CUDA call
    assert lib.pa_write_kv(NULL, NULL, NULL, 0, 1, NULL, NULL, NULL, NULL, NULL, NULL) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_write_kv(C.byref(g), NULL, NULL, 5, 1, NULL, NULL, NULL, NULL, NULL, NULL) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_write_kv(C.byref(g), NULL, NULL, 0, -1, NULL, NULL, NULL, NULL, NULL, NULL) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_write_kv(C.byref(g), NULL, NULL, 0, 0, NULL, NULL, NULL, NULL, NULL, NULL) == pa.PA_OK
    assert lib.pa_write_kv(C.byref(g), NULL, NULL, 0, 3, NULL, NULL, NULL, NULL, NULL, NULL) == pa.PA_ERR_INVALID_ARG
    # misaligned pool
    assert lib.pa_write_kv(C.byref(g), 8, 16, 0, 3, 16, 16, 32, 48, 16, NULL) == pa.PA_ERR_INVALID_ARG
    # prefill: unsupported head dim, then null pointers
    g96 = pa.geom(8, 2, 96, 1, 1, 4, 8)
    assert lib.pa_prefill(C.byref(g96), NULL, NULL, NULL, 0, 1, NULL, NULL, 4, 4, C.c_float(0.1),
                          NULL, NULL, NULL, NULL) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_prefill(C.byref(g), NULL, NULL, NULL, 0, 1, NULL, NULL, 4, 4, C.c_float(0.1),
                          NULL, NULL, NULL, NULL) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_prefill(C.byref(g), NULL, NULL, NULL, 0, 0, NULL, NULL, 4, 4, C.c_float(0.1),
                          NULL, NULL, NULL, NULL) == pa.PA_OK  # empty batch
    assert lib.pa_prefill(C.byref(g), NULL, NULL, NULL, 0, 1, NULL, NULL, 4, 4, C.c_float(float("nan")),
                          NULL, NULL, NULL, NULL) == pa.PA_ERR_INVALID_ARG
    # RoPE scatter: tables required and 16-byte aligned, max_pos >= 0
    assert lib.pa_write_kv_rope(C.byref(g), 16, 16, 0, 3, 16, 16, 32, 48, NULL, NULL, 8, 16,
                                NULL) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_write_kv_rope(C.byref(g), 16, 16, 0, 3, 16, 16, 32, 48, 64, 72, 8, 16,
                                NULL) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_write_kv_rope(C.byref(g), NULL, NULL, 0, 3, NULL, NULL, NULL, NULL, NULL, NULL, -1, NULL,
                                NULL) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_write_kv_rope(C.byref(g), NULL, NULL, 0, 0, NULL, NULL, NULL, NULL, NULL, NULL, 8, NULL,
                                NULL) == pa.PA_OK  # no rows
    # the softmax scale must be positive (the row max is taken on unscaled scores)
    for bad in (0.0, -0.125):
        assert lib.pa_prefill(C.byref(g), NULL, NULL, NULL, 0, 1, NULL, NULL, 4, 4, C.c_float(bad),
                              NULL, NULL, NULL, NULL) == pa.PA_ERR_INVALID_ARG
        assert lib.pa_decode(C.byref(g), NULL, NULL, NULL, 0, 1, NULL, NULL, 4, C.c_float(bad), NULL, NULL,
                             NULL, 0, NULL, NULL) == pa.PA_ERR_INVALID_ARG
    # backward: no rows is a no-op; bad scale, head dim, pointers and alignment are refused
    bw = lambda gg, T, sc, ptr=NULL, lse=NULL: lib.pa_prefill_backward(
        C.byref(gg), ptr, ptr, ptr, 0, 1, ptr, ptr, 4, T, C.c_float(sc), ptr, lse, ptr, lse, ptr, ptr, ptr, ptr, NULL)
    assert bw(g, 0, 0.1) == pa.PA_OK
    assert bw(g, 4, 0.0) == pa.PA_ERR_INVALID_ARG
    assert bw(g96, 4, 0.1) == pa.PA_ERR_UNSUPPORTED
    assert bw(g, 4, 0.1) == pa.PA_ERR_INVALID_ARG                  # null pointers
    assert bw(g, 4, 0.1, ptr=24, lse=16) == pa.PA_ERR_INVALID_ARG  # 8-byte aligned tensors
    assert bw(g, 4, 0.1, ptr=32, lse=18) == pa.PA_ERR_INVALID_ARG  # misaligned fp32 rows
    # decode: unsupported group size 3, too-small workspace
    g3 = pa.geom(6, 2, 64, 1, 1, 4, 8)
    assert lib.pa_decode(C.byref(g3), NULL, NULL, NULL, 0, 1, NULL, NULL, 4, C.c_float(0.1), NULL, NULL,
                         NULL, 0, NULL, NULL) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_decode(C.byref(g), 16, 16, 16, 0, 1, 16, 16, 64, C.c_float(0.1), 16, NULL, 16, 16, 16,
                         NULL) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode(C.byref(g), NULL, NULL, NULL, 0, 0, NULL, NULL, 4, C.c_float(0.1), NULL, NULL,
                         NULL, 0, NULL, NULL) == pa.PA_OK  # empty batch
    # the allocation-free decode answers the same way, before its scratch lookup (a CUDA call)
    nd = lambda gg, layer, batch, sc, ptr=NULL: lib.pa_decode_noalloc(
        gg, ptr, ptr, ptr, layer, batch, ptr, ptr, 64, C.c_float(sc), ptr, NULL, ptr, NULL)
    assert nd(NULL, 0, 1, 0.1) == pa.PA_ERR_INVALID_ARG
    assert nd(C.byref(g), 3, 1, 0.1) == pa.PA_ERR_INVALID_ARG      # layer out of range
    assert nd(C.byref(g), 0, 1, 0.0) == pa.PA_ERR_INVALID_ARG      # scale
    assert nd(C.byref(g3), 0, 1, 0.1) == pa.PA_ERR_UNSUPPORTED
    assert nd(C.byref(g), 0, 0, 0.1) == pa.PA_OK                   # empty batch
    assert nd(C.byref(g), 0, 1, 0.1) == pa.PA_ERR_INVALID_ARG      # null pointers
    assert nd(C.byref(g), 0, 1, 0.1, ptr=24) == pa.PA_ERR_INVALID_ARG  # 8-byte aligned tensors


def test_page_calls_refuse_more_slots_than_the_duplicate_check_covers(lib):
    """The page kernels keep one shared-memory bit per slot to refuse a slot
    named twice; a geometry with more slots is refused up front."""
    NULL = None
    big = pa.geom(8, 2, 64, 1, pa.PA_PAGES_MAX_SLOTS + 1, 4, 8)
    ok = pa.geom(8, 2, 64, 1, pa.PA_PAGES_MAX_SLOTS, 4, 8)
    assert lib.pa_alloc_pages(C.byref(big), 16, 1, 16, NULL, 16, 16, 16, 16, NULL) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_release_slots(C.byref(big), 16, 1, 16, 16, 16, 16, NULL) == pa.PA_ERR_UNSUPPORTED
    # at the limit the call goes on to its pointer checks (nothing enqueued here)
    assert lib.pa_alloc_pages(C.byref(ok), NULL, 1, 16, NULL, 16, 16, 16, 16, NULL) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_release_slots(C.byref(ok), NULL, 1, 16, 16, 16, 16, NULL) == pa.PA_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(ImportError):
        pa.load_library(str(tmp_path / "nope" / "libpa.so"))
