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


def test_q8_pools_check_their_shapes_and_scale_arrays(lib):
    # q8_0: whole 32-value groups per head row, and a block's scales of all
    # heads in whole 16-byte vectors; the scale arrays must be non-null,
    # 16-byte aligned, and only q8_0 pools take them
    import ctypes as C

    from paged_kv_cache_65_gb300 import PagedKVCache, _lib
    from paged_kv_cache_65_gb300._lib import KVError

    with pytest.raises(KVError):
        PagedKVCache(1, 8, 16, 2, 48, "q8_0", allocate=False)   # 48 is not 32 k
    with pytest.raises(KVError):
        PagedKVCache(1, 8, 1, 1, 32, "q8_0", allocate=False)    # 1 * 1 * 1 * 2 bytes of scales
    c = PagedKVCache(1, 8, 16, 2, 128, "q8_0", allocate=False)
    buf = (C.c_uint8 * 64)()
    base = (C.addressof(buf) + 15) & ~15
    assert lib.lib.kv_pool_set_q8_scales(c.handle, None, C.c_void_p(base)) == _lib.KV_ERR_INVALID_ARG
    assert lib.lib.kv_pool_set_q8_scales(c.handle, C.c_void_p(base + 4),
                                     C.c_void_p(base)) == _lib.KV_ERR_INVALID_ARG
    assert lib.lib.kv_pool_set_q8_scales(c.handle, C.c_void_p(base),
                                     C.c_void_p(base + 16)) == _lib.KV_OK
    bf = PagedKVCache(1, 8, 16, 2, 128, "bf16", allocate=False)
    assert lib.lib.kv_pool_set_q8_scales(bf.handle, C.c_void_p(base),
                                     C.c_void_p(base)) == _lib.KV_ERR_INVALID_ARG
