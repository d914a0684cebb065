"""Oracle q8_0 KV storage.  TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

"第 8 章 推理优化" §8.4.2 and Fig. 8-23 describe q8_0 by its bytes: every 32
values share one 2-byte scale and keep an 8-bit code each, 34 bytes where
BF16 takes 64.  The pages give no rounding rule; the reading taken here is
the plainest one the layout supports, written out step by step for one
group of 32 float32 values ``x``:

1. ``amax = max |x|``;
2. ``d = amax / 127`` in float32 (IEEE division), then the nearest fp16
   value, ties to even: the stored scale;
3. if ``d`` is 0 (an all-zero group) every code is 0; otherwise each code is
   ``x / d`` in float32 (IEEE division), rounded to the nearest integer, ties
   to even, and clamped to [-127, 127] (the fp16 rounding of ``d`` can put
   the largest ``|x| / d`` just above 127);
4. a stored value decodes as ``code * d``.

Codes are kept as int8 bit patterns (uint8 storage), scales as fp16 bit
patterns (uint16 storage).
"""

from __future__ import annotations

import numpy as np

GROUP = 32
CODE_MAX = 127


def q8_encode(x) -> tuple[np.ndarray, np.ndarray]:
    """float32 values ``[..., n]`` (n a multiple of 32) -> ``(codes uint8
    [..., n], scales uint16 [..., n / 32])``."""
    xf = np.asarray(x, dtype=np.float32)
    n = xf.shape[-1]
    if n % GROUP:
        raise ValueError("q8_0 groups hold 32 values")
    g = xf.reshape(xf.shape[:-1] + (n // GROUP, GROUP))
    amax = np.max(np.abs(g), axis=-1)                                  # step 1
    d32 = (amax / np.float32(CODE_MAX)).astype(np.float32)             # step 2
    d16 = d32.astype(np.float16)
    d = d16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d > 0, np.rint((g / d).astype(np.float32)), 0.0)  # step 3
    q = np.clip(q, -CODE_MAX, CODE_MAX).astype(np.int8)
    codes = q.reshape(xf.shape).view(np.uint8)
    return codes, d16.view(np.uint16)


def q8_decode(codes, scales) -> np.ndarray:
    """``(codes uint8 [..., n], scales uint16 [..., n / 32])`` -> float64
    values ``code * scale`` (step 4)."""
    c = np.asarray(codes, dtype=np.uint8).view(np.int8).astype(np.float64)
    s = np.asarray(scales, dtype=np.uint16).view(np.float16).astype(np.float64)
    n = c.shape[-1]
    return (c.reshape(c.shape[:-1] + (n // GROUP, GROUP)) * s[..., None]).reshape(c.shape)
