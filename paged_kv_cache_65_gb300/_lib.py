"""ctypes binding of ``libpagedkv.so`` (C ABI in ``include/pagedkv.h``).

Argument marshalling only: every step of the hot path runs in the library.
Functions keep the C names; device pointers are passed as integers (for
example ``tensor.data_ptr()``), host arrays as NumPy arrays, streams as the
integer handle of a CUDA stream (``torch.cuda.current_stream().cuda_stream``)
or 0 for the legacy default stream.

Importing this module raises ``ImportError`` when the library has not been
built: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes as C
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpagedkv.so")

KV_OK = 0
KV_ERR_NO_FREE_BLOCK = 1
KV_ERR_INVALID_ARG = 2
KV_ERR_REFCOUNT = 3
KV_ERR_CUDA = 4
KV_ERR_DEVICE_CHECK = 5
KV_ERR_UNSUPPORTED = 6
KV_ERR_SCRATCH_TOO_SMALL = 7
KV_OPT_DECODE_PATH = 1
KV_OPT_PDL = 2
KV_OPT_PLAN_GRID = 3
KV_DTYPE_F32 = 0
KV_DTYPE_BF16 = 1
KV_DTYPE_FP8_E4M3 = 2
KV_DTYPE_Q8_0 = 3
# bits of the device status word
KV_DEV_BAD_BLOCK_ID = 1
KV_DEV_BAD_SLOT = 2
KV_DEV_BAD_COW_PAIR = 4
KV_DEV_WAIT_TIMEOUT = 8
KV_DEV_BAD_CONTEXT = 16
KV_DEV_SMEM_ALIGN = 32

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing; build it with `python paged_kv_cache_65_gb300/build.py` "
        "(or __graft_entry__.build())")

lib = C.CDLL(LIB_PATH)

_i32p = C.POINTER(C.c_int32)
_i64p = C.POINTER(C.c_int64)
_ip = C.POINTER(C.c_int)
_vp = C.c_void_p
_f32p = C.POINTER(C.c_float)

# (name, restype, argtypes): every symbol declared in include/pagedkv.h
SIGNATURES = [
    ("kv_status_string", C.c_char_p, [C.c_int]),
    ("kv_pool_create", C.c_int, [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, _vp, _vp,
                                 _vp, _i32p, C.POINTER(_vp)]),
    ("kv_pool_destroy", None, [_vp]),
    ("kv_pool_stats", C.c_int, [_vp, _ip, _ip, _ip]),
    ("kv_pool_check", C.c_int, [_vp]),
    ("kv_block_refcount", C.c_int, [_vp, C.c_int32, _ip]),
    ("kv_pool_set_option", C.c_int, [_vp, C.c_int, C.c_int]),
    ("kv_pool_set_fp8_scales", C.c_int, [_vp, C.c_float, C.c_float]),
    ("kv_pool_set_q8_scales", C.c_int, [_vp, _vp, _vp]),
    ("kv_pool_device_status", C.c_int, [_vp, _vp, _ip]),
    ("kv_device_wait_selftest", C.c_int, [_vp, C.c_int, _vp]),
    ("block_alloc", C.c_int, [_vp, C.c_int, _i32p]),
    ("block_free", C.c_int, [_vp, _i32p, C.c_int]),
    ("block_fork", C.c_int, [_vp, _i32p, C.c_int]),
    ("block_cow", C.c_int, [_vp, C.c_int32, _i32p]),
    ("seq_append_slots", C.c_int, [_vp, _i32p, C.c_int, _i64p, _i32p, _ip]),
    ("seq_append_tokens", C.c_int, [_vp, C.c_int32, C.c_int, _i64p, _i32p, _ip]),
    ("seq_fork", C.c_int, [_vp, C.c_int32, C.c_int32]),
    ("seq_release", C.c_int, [_vp, C.c_int32]),
    ("kv_prefix_cache_enable", C.c_int, [_vp, C.c_uint64]),
    ("seq_match_prefix", C.c_int, [_vp, C.c_int32, _i32p, C.c_int, _ip]),
    ("seq_append_slots_ids", C.c_int, [_vp, _i32p, C.c_int, _i32p, _i64p, _i32p, _ip]),
    ("seq_append_tokens_ids", C.c_int, [_vp, C.c_int32, C.c_int, _i32p, _i64p, _i32p, _ip]),
    ("kv_prefix_evict", C.c_int, [_vp, C.c_int, _ip]),
    ("kv_prefix_stats", C.c_int, [_vp, _ip, _ip]),
    ("seq_length", C.c_int, [_vp, C.c_int32, _ip]),
    ("seq_block_table", C.c_int, [_vp, _i32p, C.c_int, C.c_int, _i32p, _i32p]),
    ("cow_copy", C.c_int, [_vp, _vp, C.c_int, _vp]),
    ("reshape_and_cache", C.c_int, [_vp, C.c_int, _vp, _vp, _vp, C.c_int, _vp]),
    ("paged_decode_workspace_bytes", C.c_size_t, [_vp, C.c_int, C.c_int]),
    ("paged_decode_partials", C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, C.c_int, _vp, C.c_int,
                                        C.c_float, _vp, C.c_size_t, _vp]),
    ("paged_decode_merge", C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, C.c_int, _vp, C.c_size_t,
                                     _vp]),
    ("paged_decode_attention", C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, C.c_int, _vp, C.c_int,
                                         C.c_float, _vp, C.c_int, _vp, C.c_size_t, _vp]),
    ("paged_decode_plan_bytes", C.c_size_t, [_vp, C.c_int, C.c_int]),
    ("paged_decode_plan", C.c_int, [_vp, _i32p, C.c_int, C.c_int, C.c_int, C.c_int, _vp,
                                    C.c_size_t, C.POINTER(C.c_size_t)]),
    ("paged_decode_partials_planned", C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, C.c_int, _vp,
                                                _vp, C.c_float, _vp, C.c_size_t, _vp]),
    ("paged_decode_merge_planned", C.c_int, [_vp, C.c_int, _vp, _vp, _vp, C.c_int, _vp,
                                             C.c_size_t, _vp]),
    ("paged_decode_partials_planned_write", C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, _vp, _vp,
                                                      C.c_int, _vp, _vp, C.c_float, _vp,
                                                      C.c_size_t, _vp]),
    ("paged_decode_attention_planned", C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, C.c_int, _vp,
                                                 _vp, C.c_float, _vp, C.c_int, _vp, C.c_size_t,
                                                 _vp]),
    ("paged_decode_attention_noalloc", C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, C.c_int, _vp,
                                                 C.c_int, C.c_float, _vp, C.c_int, _vp]),
    ("paged_prefill_attention", C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, C.c_int, _vp, _vp,
                                          C.c_int, C.c_int, C.c_float, _vp, C.c_int, _vp]),
    ("paged_prefill_schedule_bytes", C.c_size_t, [_vp, C.c_int, C.c_int, C.c_int]),
    ("paged_prefill_schedule", C.c_int, [_vp, _i32p, _i32p, C.c_int, C.c_int, _vp, C.c_size_t,
                                         C.POINTER(C.c_int)]),
    ("paged_prefill_attention_scheduled", C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, C.c_int,
                                                    _vp, _vp, C.c_int, _vp, C.c_int, C.c_float,
                                                    _vp, C.c_int, _vp]),
    ("paged_prefill_staging_bytes", C.c_size_t, [_vp, C.c_int, C.c_int]),
    ("paged_prefill_attention_staged", C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, C.c_int, _vp,
                                                 _vp, C.c_int, C.c_int, _vp, C.c_int, C.c_float,
                                                 _vp, C.c_int, _vp, C.c_size_t, _vp]),
    ("kv_decode_step_staging_bytes", C.c_size_t, [_vp, C.c_int, C.c_int, C.c_int]),
    # the host buffers go as plain addresses (the per-step call is marshalled
    # with as few conversions as possible)
    ("kv_decode_step_host", C.c_int, [_vp, _vp, C.c_int, C.c_int, C.c_int, _vp, _vp, _vp,
                                      C.c_float, _vp, _vp, C.c_size_t, _vp]),
]

for _name, _res, _args in SIGNATURES:
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class KVError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        msg = lib.kv_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})" if where else msg)


def check(status: int, where: str = "") -> None:
    if status != KV_OK:
        raise KVError(status, where)


def i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def ptr_i32(a: np.ndarray):
    return a.ctypes.data_as(_i32p)


def ptr_i64(a: np.ndarray):
    return a.ctypes.data_as(_i64p)


def ptr_f32(a: np.ndarray):
    return a.ctypes.data_as(_f32p)


def vp(x) -> _vp:
    """A device/host address from an int, a torch tensor or a NumPy array."""
    if x is None:
        return _vp(0)
    if isinstance(x, int):
        return _vp(x)
    if hasattr(x, "data_ptr"):
        return _vp(x.data_ptr())
    if isinstance(x, np.ndarray):
        return _vp(x.ctypes.data)
    raise TypeError(type(x))
