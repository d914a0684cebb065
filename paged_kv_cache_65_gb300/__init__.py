"""GB300-native paged KV cache: decode attention over a paged KV cache,
its per-step slot write, the copy-on-write block copy, and the ref-counted
free-list block manager, behind the C ABI of ``include/pagedkv.h``.

The compute path is ``libpagedkv.so`` (CUDA for sm_103a plus the C++ block
manager).  This package only marshals arguments; importing it fails when the
library has not been built.
"""

from . import _lib  # noqa: F401  (raises ImportError when the library is missing)
from ._lib import KVError, SIGNATURES, lib  # noqa: F401
from .cache import PagedKVCache  # noqa: F401

__all__ = ["PagedKVCache", "KVError", "lib", "SIGNATURES"]
