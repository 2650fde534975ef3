"""The C-ABI library builds, loads without a GPU and exports every entry point
include/pa.h declares; host-side argument checks answer without a device."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_72_gb300 import _lib
from paged_kv_cache_72_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    decls = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pa_\w+)\s*\(([^;]*)\);", text, flags=re.M)
    out = {}
    for name, args in decls:
        args = args.strip()
        out[name] = 0 if args in ("", "void") else len(args.split(","))
    return out


def test_binding_constants_match_the_header():
    # every value #define in the header has the same value in the binding
    text = open(HEADER).read()
    found = 0
    for name, val in re.findall(r"^#define[ \t]+(PA_\w+)[ \t]+(\S.*?)[ \t]*(?:/\*.*)?$", text, flags=re.M):
        expr = val.replace("u", "")
        assert hasattr(_lib, name), name
        assert getattr(_lib, name) == eval(expr, {}), (name, val)
        found += 1
    assert found >= 19


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def test_header_declares_the_entry_points():
    names = set(_declared())
    assert {"pa_cache_write", "pa_decode", "pa_copy_blocks", "pa_slot_mapping",
            "pa_decode_workspace_size", "pa_gather_kv", "pa_get_error", "pa_strerror",
            "pa_version"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name, nargs in _declared().items():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, name
        assert len(_lib.SIGNATURES[name][1]) == nargs, (name, nargs)


def test_strerror_and_version(lib):
    assert lib.pa_version() >= 100
    for code in range(6):
        assert lib.pa_strerror(code)
    assert lib.pa_strerror(99) == b"unknown status"


def test_host_checks_need_no_device(lib):
    n = ctypes.c_size_t(0)
    # unsupported head_dim / block size / group size are refused before any CUDA call
    assert lib.pa_decode_workspace_size(8, 8, 96, 16, 0, 0, 0, ctypes.byref(n)) == 2
    assert lib.pa_decode_workspace_size(8, 8, 128, 12, 0, 0, 0, ctypes.byref(n)) == 2
    assert lib.pa_decode_workspace_size(8, 8, 128, 1, 0, 0, 0, ctypes.byref(n)) == 2
    assert lib.pa_decode_workspace_size(64, 2, 128, 16, 0, 0, 0, ctypes.byref(n)) == 2
    assert lib.pa_decode_workspace_size(6, 4, 128, 16, 0, 0, 0, ctypes.byref(n)) == 1
    assert lib.pa_decode_workspace_size(8, 8, 128, 16, 7, 0, 0, ctypes.byref(n)) == 2
    assert lib.pa_decode_workspace_size(8, 8, 128, 16, 0, 0, 0, None) == 1
    # an E4M3 cache whose chunk would need more than 32 TMA boxes (32 tokens
    # per warp, one KV head per group, 4-token blocks) is refused
    assert lib.pa_decode_workspace_size(6, 3, 64, 4, 2, 0, 0, ctypes.byref(n)) == 2
    # a grid beyond the fixed counter region is refused
    assert lib.pa_decode_workspace_size(8, 8, 128, 16, 0, 0, _lib.PA_DECODE_MAX_CTAS + 1,
                                        ctypes.byref(n)) == 1
    # empty batches are no-ops
    assert lib.pa_cache_write(None, None, None, 0, None, None, 10, 16, 8, 128, 0, None, None) == 0
    assert lib.pa_copy_blocks(None, 0, None, None, 10, 16, 8, 128, 0, None, None) == 0
    assert lib.pa_slot_mapping(None, 4, 2, None, None, 0, 16, 10, None, None, None) == 0
    # missing pointers and negative sizes
    assert lib.pa_cache_write(None, None, None, 3, None, None, 10, 16, 8, 128, 0, None, None) == 1
    assert lib.pa_cache_write(None, None, None, -1, None, None, 10, 16, 8, 128, 0, None, None) == 1
    # the slot-mapped cache write: no tokens is a no-op, missing inputs or a
    # negative count are refused, E4M3 pools are not its dtype
    assert lib.pa_cache_write_mapped(None, None, None, 4, 2, None, None, 0, None, None, 10, 16, 8,
                                     128, 0, None, None, None) == 0
    assert lib.pa_cache_write_mapped(None, None, None, 4, 2, None, None, 3, None, None, 10, 16, 8,
                                     128, 0, None, None, None) == 1
    assert lib.pa_cache_write_mapped(None, None, None, 4, 2, None, None, -1, None, None, 10, 16, 8,
                                     128, 0, None, None, None) == 1
    assert lib.pa_cache_write_mapped(None, None, None, 4, 2, None, None, 3, None, None, 10, 16, 8,
                                     128, 2, None, None, None) == 2
    assert lib.pa_cache_write_fp8_mapped(None, None, 1, None, 4, 2, None, None, 0, None, None, 10,
                                         16, 8, 128, 1.0, 1.0, None, None, None) == 0
    assert lib.pa_cache_write_fp8_mapped(None, None, 1, None, 4, 2, None, None, 3, None, None, 10,
                                         16, 8, 128, 1.0, 1.0, None, None, None) == 1
    assert lib.pa_cache_write_fp8_mapped(None, None, 1, None, 4, 2, None, None, 3, None, None, 10,
                                         16, 8, 128, 0.0, 1.0, None, None, None) == 1
    assert lib.pa_get_error(None, None, None) == 1
