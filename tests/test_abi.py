"""The C-ABI library loads here (no GPU needed) and exports every symbol
that ``include/pagedkv.h`` declares; the Python binding covers the same set."""

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "pagedkv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^(?:kvStatus|void|size_t|const char\*)\s+(\w+)\s*\(", text, flags=re.M))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_65_gb300 import _lib

    return _lib


def test_header_declares_the_pool_block_and_kernel_calls():
    names = declared_functions()
    for n in ("kv_pool_create", "block_alloc", "block_free", "block_fork", "block_cow",
              "reshape_and_cache", "paged_decode_attention", "cow_copy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in sorted(names):
        assert hasattr(lib.lib, n), f"{n} not exported"
    assert {s[0] for s in lib.SIGNATURES} == names


def test_status_strings(lib):
    assert lib.lib.kv_status_string(0) == b"ok"
    assert lib.lib.kv_status_string(1) == b"no free KV block"


def test_device_calls_fail_cleanly_on_host_only_pool(lib):
    from paged_kv_cache_65_gb300 import PagedKVCache, KVError

    c = PagedKVCache(1, 8, 4, 2, 64, "f32", allocate=False)
    with pytest.raises(KVError) as e:
        c.reshape_and_cache(0, 16, 16, 16, 1)
    assert e.value.status == lib.KV_ERR_INVALID_ARG
    assert c.paged_decode_workspace_bytes(4, 8) > 0
    assert c.paged_decode_workspace_bytes(4, 7) == 0  # H_q not a multiple of H_kv
