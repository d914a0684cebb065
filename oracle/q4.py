"""Oracle q4_0 group codes.  TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

"第 8 章 推理优化" §8.4.2 and Fig. 8-23 describe q4_0 by its bytes: every 32
values share one 2-byte scale and keep a 4-bit code each, 18 bytes where
BF16 takes 64.  The pages give neither a rounding rule nor a nibble order;
the reading taken here is the plainest one the layout supports, the q8_0
rule of ``oracle/q8.py`` with 7 in place of 127, for one group of 32 float32
values ``x``:

1. ``amax = max |x|``;
2. ``d = amax / 7`` in float32 (IEEE division), then the nearest fp16 value,
   ties to even: the stored scale;
3. if ``d`` is 0 (an all-zero group) every code is 0; otherwise each code is
   ``x / d`` in float32 (IEEE division), rounded to the nearest integer, ties
   to even, and clamped to [-7, 7];
4. a code ``c`` is stored as the nibble ``c + 8`` (1 .. 15; 8 is zero), two
   values a byte: value ``2i`` in the low nibble of byte ``i``, value
   ``2i + 1`` in its high nibble;
5. a stored value decodes as ``c * d``.

Packed codes are uint8 ``[..., n / 2]``, scales fp16 bit patterns (uint16)
``[..., n / 32]``.
"""

from __future__ import annotations

import numpy as np

GROUP = 32
CODE_MAX = 7
OFFSET = 8


def q4_codes(x) -> tuple[np.ndarray, np.ndarray]:
    """float32 values ``[..., n]`` (n a multiple of 32) -> ``(signed codes
    int8 [..., n] in [-7, 7], scales uint16 [..., n / 32])`` (steps 1-3)."""
    xf = np.asarray(x, dtype=np.float32)
    n = xf.shape[-1]
    if n % GROUP:
        raise ValueError("q4_0 groups hold 32 values")
    g = xf.reshape(xf.shape[:-1] + (n // GROUP, GROUP))
    amax = np.max(np.abs(g), axis=-1)                                  # step 1
    d32 = (amax / np.float32(CODE_MAX)).astype(np.float32)             # step 2
    d16 = d32.astype(np.float16)
    d = d16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d > 0, np.rint((g / d).astype(np.float32)), 0.0)  # step 3
    q = np.clip(q, -CODE_MAX, CODE_MAX).astype(np.int8)
    return q.reshape(xf.shape), d16.view(np.uint16)


def q4_pack(codes) -> np.ndarray:
    """Signed codes int8 ``[..., n]`` -> bytes uint8 ``[..., n / 2]`` (step 4)."""
    c = np.asarray(codes, dtype=np.int16) + OFFSET
    lo, hi = c[..., 0::2], c[..., 1::2]
    return (lo | (hi << 4)).astype(np.uint8)


def q4_unpack(packed) -> np.ndarray:
    """Bytes uint8 ``[..., n / 2]`` -> signed codes int8 ``[..., n]``."""
    b = np.asarray(packed, dtype=np.uint8).astype(np.int16)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.int16)
    out[..., 0::2] = (b & 0x0F) - OFFSET
    out[..., 1::2] = (b >> 4) - OFFSET
    return out.astype(np.int8)


def q4_encode(x) -> tuple[np.ndarray, np.ndarray]:
    """float32 values -> ``(packed codes uint8 [..., n / 2], scales uint16
    [..., n / 32])``."""
    codes, scales = q4_codes(x)
    return q4_pack(codes), scales


def q4_decode(packed, scales) -> np.ndarray:
    """``(packed codes, scales)`` -> float64 values ``c * d`` (step 5)."""
    c = q4_unpack(packed).astype(np.float64)
    s = np.asarray(scales, dtype=np.uint16).view(np.float16).astype(np.float64)
    n = c.shape[-1]
    return (c.reshape(c.shape[:-1] + (n // GROUP, GROUP)) * s[..., None]).reshape(c.shape)
