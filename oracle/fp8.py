"""Oracle FP8 (E4M3) KV storage.  TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

"第 8 章 推理优化" §8.4.2 compares BF16 KV with narrower KV formats (an FP8
KV cache in its H100 inter-token-latency fit; q8_0 and q4_0 with a shared
scale per group of 32 values) and charges the read savings against the
conversion time.  This build's quantized pool stores each K or V element
as one FP8 E4M3 code of ``x / scale``, one float32 scale per pool for K and
one for V, so a token row costs half of BF16 (32 of every 64 bytes).

E4M3 as written here (the "FN" variant: no infinities): a sign bit, four
exponent bits with bias 7 and three mantissa bits.

* exponent field ``E`` in 1..15, mantissa ``M``: ``(1 + M / 8) * 2^(E - 7)``,
  except ``E = 15, M = 7``, which is NaN; the largest finite value is
  ``1.75 * 2^8 = 448``;
* ``E = 0``: ``M * 2^-9`` (subnormals; the smallest is ``2^-9``).

Encoding (``e4m3_encode``): ``v = x / scale`` in float32 (IEEE division),
then the nearest E4M3 value, ties to the even mantissa; magnitudes above
448, infinities included, saturate to 448 with their sign; NaN becomes the
NaN code ``0x7F`` with the input's sign.  Every step is exact float64
arithmetic on powers of two, so the encoder is a direct statement of the
rounding rule, not an approximation.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def e4m3_decode(codes) -> np.ndarray:
    """Codes (uint8) -> their values as float64 (NaN for the NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def _encode_magnitude(a: float) -> int:
    """Non-negative finite float64 -> 7-bit E4M3 magnitude code."""
    if a >= E4M3_MAX:
        return 0x7E
    if a < 2.0 ** -6:
        n = int(np.rint(a / 2.0 ** -9))  # subnormal grid, ties to even
        # n == 8 is the smallest normal, which is code 0x08 as well
        return n
    e = int(np.floor(np.log2(a)))
    # guard the floor against log2 rounding at exact powers of two
    if 2.0 ** e > a:
        e -= 1
    elif 2.0 ** (e + 1) <= a:
        e += 1
    q = 2.0 ** (e - 3)  # spacing of the values in [2^e, 2^(e+1))
    n = int(np.rint(a / q))  # 8..16, ties to even
    if n == 16:
        n, e = 8, e + 1
    if e > 8 or (e == 8 and n > 14):  # beyond 448
        return 0x7E
    return ((e + 7) << 3) | (n - 8)


def e4m3_encode(x, scale: float = 1.0) -> np.ndarray:
    """float32 values (any shape) -> uint8 codes of ``x / scale``."""
    xf = np.asarray(x, dtype=np.float32)
    v = (xf / np.float32(scale)).astype(np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    flat_v, flat_o = v.reshape(-1), out.reshape(-1)
    for i in range(flat_v.size):
        f = float(flat_v[i])
        neg = bool(np.signbit(flat_v[i]))
        if np.isnan(f):
            code = NAN_CODE
        else:
            code = _encode_magnitude(abs(f))
        flat_o[i] = code | (0x80 if neg else 0)
    return out
