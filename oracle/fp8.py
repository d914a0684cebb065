"""Oracle FP8 (E4M3) KV storage.  TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

"第 8 章 推理优化" §8.4.2 compares BF16 KV with narrower KV formats (an FP8
KV cache in its H100 inter-token-latency fit; q8_0 and q4_0 with a shared
scale per group of 32 values) and charges the read savings against the
conversion time.  The FP8 pool modelled here stores each K or V element
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


def e4m3_encode(x, scale: float = 1.0) -> np.ndarray:
    """float32 values (any shape) -> uint8 codes of ``x / scale``."""
    xf = np.asarray(x, dtype=np.float32)
    v = (xf / np.float32(scale)).astype(np.float32)
    a = np.abs(v).astype(np.float64)  # exact
    nan = np.isnan(v)
    code = np.zeros(v.shape, dtype=np.int64)
    # below the smallest normal: the nearest multiple of 2^-9 (ties to even);
    # 8 * 2^-9 = 2^-6 is the smallest normal, whose code is 0x08 as well
    sub = ~nan & (a < 2.0 ** -6)
    code[sub] = np.rint(a[sub] / 2.0 ** -9)
    # normal range: a in [2^e, 2^(e+1)), spacing 2^(e-3), ties to even
    nrm = ~nan & ~sub & (a < E4M3_MAX)
    an = a[nrm]
    e = np.floor(np.log2(an))
    e -= np.exp2(e) > an  # guard the floor against log2 rounding
    e += np.exp2(e + 1) <= an
    n = np.rint(an / np.exp2(e - 3))  # 8 .. 16
    carry = n == 16
    n[carry] = 8
    e[carry] += 1
    c = ((e.astype(np.int64) + 7) << 3) | (n.astype(np.int64) - 8)
    c[(e > 8) | ((e == 8) & (n > 14))] = 0x7E  # rounded beyond 448
    code[nrm] = c
    code[~nan & (a >= E4M3_MAX)] = 0x7E  # saturation, infinities included
    code[nan] = NAN_CODE
    code |= np.where(np.signbit(v), 0x80, 0)
    return code.astype(np.uint8)
