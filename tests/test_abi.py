"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/mla.h declares, and rejects bad arguments before any
CUDA call."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build_library()
    return ctypes.CDLL(path)


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(mla_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["mla_absorb_weights", "mla_cache_append", "mla_decode", "mla_decode_workspace_bytes",
                     "mla_get_device_status", "mla_cache_page_bytes"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_page_bytes(lib):
    lib.mla_cache_page_bytes.restype = ctypes.c_size_t
    assert lib.mla_cache_page_bytes(0) == 64 * 1152
    assert lib.mla_cache_page_bytes(1) == 64 * 624
    assert lib.mla_cache_page_bytes(2) == 64 * 400
    # the quantizer variants write the INT8 / INT4 page layouts
    assert lib.mla_cache_page_bytes(3) == 64 * 624
    assert lib.mla_cache_page_bytes(4) == 64 * 400
    assert lib.mla_cache_page_bytes(5) == 64 * 400
    assert lib.mla_cache_page_bytes(6) == 0
    assert lib.mla_cache_page_bytes(7) == 0


def test_host_validation_without_gpu(lib):
    import mla_absorbed_latent_gb300 as m
    raw = m.raw_library()
    assert raw.mla_absorb_weights(None, 7, None, None, None) == m.MLA_ERR_UNSUPPORTED
    assert raw.mla_absorb_weights(None, 16, None, None, None) == m.MLA_ERR_INVALID
    assert raw.mla_absorb_weights(24, 16, 32, 48, None) == m.MLA_ERR_INVALID   # misaligned
    bad_fmt = m.mla_cache_t(9, 1, 1024)
    assert raw.mla_cache_append(ctypes.byref(bad_fmt), None, None, None, 1, None, 1, 1, None) == m.MLA_ERR_UNSUPPORTED
    cache = m.mla_cache_t(0, 1, 1024)
    assert raw.mla_cache_append(ctypes.byref(cache), None, None, None, 1, None, -1, 1, None) == m.MLA_ERR_INVALID
    assert raw.mla_cache_append(ctypes.byref(cache), None, None, None, 1, None, 0, 5, None) == m.MLA_OK
    unaligned = m.mla_cache_t(0, 1, 1024 + 16)
    assert raw.mla_cache_append(ctypes.byref(unaligned), None, None, None, 1, None, 1, 1, None) == m.MLA_ERR_INVALID
    assert raw.mla_decode(None, None, None, None, 12, ctypes.byref(cache), None, 1, None, 1, 0.1, None, 0, None,
                          None) == m.MLA_ERR_UNSUPPORTED
    assert raw.mla_decode_workspace_bytes(-1, 128) == 0
    assert raw.mla_decode_workspace_bytes(4, 3) == 0
    # the fused producer: hidden must be whole 64-wide chunks; empty batches enqueue nothing
    proj = raw.mla_cache_project_append
    assert proj(ctypes.byref(cache), None, 100, None, None, 1e-6, 1e4, None, 1, None, 1, 1, None, 0, None, 0,
                None) == m.MLA_ERR_UNSUPPORTED
    assert proj(ctypes.byref(bad_fmt), None, 2048, None, None, 1e-6, 1e4, None, 1, None, 1, 1, None, 0, None, 0,
                None) == m.MLA_ERR_UNSUPPORTED
    assert proj(None, None, 2048, None, None, 1e-6, 1e4, None, 1, None, 1, 1, None, 0, None, 0,
                None) == m.MLA_ERR_INVALID
    assert proj(ctypes.byref(cache), None, 2048, None, None, 1e-6, 1e4, None, 1, None, 1, 1, None, -1, None, 0,
                None) == m.MLA_ERR_INVALID
    assert proj(ctypes.byref(cache), None, 2048, None, None, 1e-6, 1e4, None, 1, None, 0, 7, None, 0, None, 0,
                None) == m.MLA_OK
    assert proj(ctypes.byref(cache), None, 2048, None, None, 1e-6, 1e4, None, 1, None, 2, 1, None, 0, None, 0,
                None) == m.MLA_ERR_INVALID   # null inputs
    # the no-allocation decode checks its arguments like mla_decode, before any CUDA call
    fake = 1 << 20  # a non-null, aligned stand-in address (never dereferenced: the checks fail first)
    for bad_scale in (-1.0, 0.0, float("inf"), float("nan")):
        with pytest.raises(m.MLAError) as e:
            m.mla_decode_noalloc(fake, fake, fake, fake, 16, cache, fake, 1, fake, 1, bad_scale, fake, stream=0)
        assert e.value.status == m.MLA_ERR_INVALID
    with pytest.raises(m.MLAError) as e:
        m.mla_decode_noalloc(fake, fake, fake, fake, 12, cache, fake, 1, fake, 1, 0.07, fake, stream=0)
    assert e.value.status == m.MLA_ERR_UNSUPPORTED
    m.mla_decode_noalloc(None, None, None, None, 16, cache, None, 1, None, 0, 0.07, None, stream=0)  # B = 0
    assert raw.mla_cache_project_workspace_bytes(1, 1, 100, 0) == 0
    assert raw.mla_cache_project_workspace_bytes(-1, 1, 2048, 0) == 0


def test_status_strings(lib):
    import mla_absorbed_latent_gb300 as m
    for st in range(0, -7, -1):
        assert m.mla_status_string(st) != "unknown status"
    assert m.mla_status_string(-99) == "unknown status"
