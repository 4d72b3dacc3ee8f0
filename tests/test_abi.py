"""The C-ABI library builds, loads and exports everything include/hs.h declares.

These run without a GPU: only argument checks that return before any CUDA call.
"""
import os
import re

import numpy as np
import pytest

import hierarchical_kv_cache_swap_gb300 as hs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hs.h")


@pytest.fixture(scope="module")
def lib():
    hs.build()
    return hs.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(hs_[a-z_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("hs_create", "hs_resolve", "hs_destroy"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(hs.SIGNATURES), "binding and header disagree"
    for n in names:
        assert hasattr(lib, n), n


def test_library_is_built_for_sm_103a():
    text = open(os.path.join(ROOT, "hierarchical_kv_cache_swap_gb300", "_nvcc.py")).read()
    assert "arch=compute_103a,code=sm_103a" in text


def test_create_rejects_bad_sizes_before_touching_cuda(lib):
    assert not lib.hs_create(0, 8, 8, 16)
    assert "positive" in hs.last_error()
    assert not lib.hs_create(1, 8, 8, 24)
    assert "multiple of 16" in hs.last_error()
    assert not lib.hs_create(1, 8, 70000, 16)
    assert "exceeds" in hs.last_error()
    assert not lib.hs_create(2_000_000, 8, 8, 16)
    assert "exceeds" in hs.last_error()
    assert not lib.hs_create(1 << 14, 1 << 10, 1 << 14, 1 << 12)
    assert "32 GiB" in hs.last_error()


def test_lent_host_store_is_validated_before_touching_cuda(lib):
    import ctypes
    buf = (ctypes.c_uint8 * 4096)()
    addr = ctypes.addressof(buf)
    assert not lib.hs_create_with_host(1, 8, 8, 16, None, 16)
    assert "16-byte aligned" in hs.last_error()
    assert not lib.hs_create_with_host(1, 8, 8, 32, (addr + 15) & ~15, 16)   # stride < E
    assert not lib.hs_create_with_host(1, 8, 8, 16, ((addr + 15) & ~15) + 8, 16)  # misaligned
    assert lib.hs_checksum_rows(None, None, None, 1, 1, None) == hs.HS_ERR_INVALID


def test_calls_on_null_context_fail_cleanly(lib):
    assert lib.hs_resolve(None, None, None, 1, 1, None, None) == hs.HS_ERR_INVALID
    assert lib.hs_resolve_host(None, None, None, 1, 1, None, None) == hs.HS_ERR_INVALID
    assert lib.hs_set_flags(None, 0) == hs.HS_ERR_INVALID
    assert lib.hs_set_wait_limit(None, 1_000_000) == hs.HS_ERR_INVALID
    assert lib.hs_reset(None, None) == hs.HS_ERR_INVALID
    assert lib.hs_kernels_per_call(None) == hs.HS_ERR_INVALID
    assert lib.hs_host_kv(None) is None and lib.hs_host_stride(None) == 0
    lib.hs_destroy(None)


def test_binding_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(hs.HsError):
        hs.load_library(str(tmp_path / "missing.so"))


def test_addr_of_numpy_arrays_matches_ctypes_data():
    """The binding's fast address path agrees with numpy's own for every kind of array."""
    a = np.arange(64, dtype=np.int32).reshape(8, 8)
    ro = a.copy()
    ro.flags.writeable = False
    cases = [a, a[3], a[2:5], a[:, 1], ro, ro[2], np.empty(0, np.int32), np.empty((0, 4), np.int32)]
    for x in cases:
        assert hs._addr(x) == x.ctypes.data


def test_resolve_host_rejects_bad_buffers_before_any_call():
    """The host-buffer entry point's binding checks dtype, layout and shapes before it
    reaches the library (so no context, and no GPU, is needed to exercise them)."""
    ctx = object.__new__(hs.Context)
    sel = np.zeros((2, 4), np.int32)
    out = np.zeros((2, 4), np.int32)
    miss = np.zeros(2, np.int32)
    bad = [
        (sel.astype(np.int64), out, miss),            # wrong dtype
        (sel, np.zeros((2, 8), np.int32)[:, ::2], miss),  # not contiguous
        (sel, np.zeros((2, 3), np.int32), miss),      # out_slots shape
        (sel, out, np.zeros(3, np.int32)),            # miss_counts shape
        (sel.tolist(), out, miss),                    # not an array
    ]
    for args in bad:
        with pytest.raises(ValueError):
            ctx.resolve_host(*args)
