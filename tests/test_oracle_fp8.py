"""Pins of the quantized-KV oracle: the pages' byte arithmetic for narrower KV
formats ("第 8 章 推理优化" §8.4.2, Fig. 8-23), the E4M3 code table fixed by the
format's definition, nearest-value rounding checked by brute force against
that table, and the FP8 pool's write / copy / gather behaviour."""

import math

import numpy as np
import pytest

from oracle.attention import decode_attention
from oracle.fp8 import e4m3_decode, e4m3_encode
from oracle.kv_store import KVStore
from oracle.sizing import GROUP32_BYTES, bits_per_value, fit_crossover, quantized_bytes, read_saving


# ---------------------------------------------------------------- the pages


def test_quantized_sizes_printed_on_the_pages(golden):
    g = golden("kv_quant_examples.json")
    for ex in g["sizes_mib"]:
        assert quantized_bytes(ex["bf16"], ex["fmt"]) == ex["mib"], ex["cite"]
    sv = g["savings_mib"]
    for fmt in ("q8_0", "q4_0"):
        assert sv["bf16"] - quantized_bytes(sv["bf16"], fmt) == sv[fmt], sv["cite"]
    gb = g["group_bytes"]
    for fmt in ("bf16", "q8_0", "q4_0"):
        assert GROUP32_BYTES[fmt] == gb[fmt], gb["cite"]
    bpv = g["bits_per_value"]
    for fmt in ("q8_0", "q4_0"):
        assert bits_per_value(fmt) == bpv[fmt], bpv["cite"]
    r = g["sixteen_requests_gib"]
    total = r["requests"] * r["mib_each"] / 1024
    assert round(total, 2) == r["gib"] and total < r["budget_gib"], r["cite"]


def test_read_saving_examples(golden):
    ex = golden("kv_quant_examples.json")["read_saving_ms"]
    beta = ex["peak_gbs"] * 1e9 * ex["efficiency"]  # bytes per second
    saved_ms = read_saving(ex["delta_mib"] * 2 ** 20, beta, 0.0) * 1e3
    # the page rounds its bandwidth to "about 1.16 TB/s"
    assert abs(saved_ms - ex["saving"]) < 2e-3, ex["cite"]
    for t_c, net in ex["cases"]:
        assert abs(read_saving(ex["delta_mib"] * 2 ** 20, beta, t_c * 1e-3) * 1e3 - net) < 2e-3


def test_itl_fit_crossover(golden):
    ex = golden("kv_quant_examples.json")["itl_fit"]
    (a0, b0), (a1, b1) = ex["bf16"], ex["fp8"]
    assert round(fit_crossover(a0, b0, a1, b1), -2) == ex["crossover"], ex["cite"]
    for L, t_bf16, t_fp8 in ex["points"]:
        assert round(a0 + b0 * L, 2) == t_bf16 and round(a1 + b1 * L, 2) == t_fp8


def test_fp8_pool_halves_the_bf16_bytes():
    # one scale per pool: 32 of every 64 bytes, below q8_0's 34
    assert quantized_bytes(1152, "fp8_e4m3") == 576
    assert bits_per_value("fp8_e4m3") == 8


# ------------------------------------------------------------- E4M3 codes

# values the E4M3 definition fixes (sign, 4-bit exponent with bias 7, 3-bit
# mantissa, no infinities, NaN = exponent and mantissa all ones)
DEFINED = [
    (0x00, 0.0), (0x80, -0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x30, 0.5), (0x38, 1.0), (0x39, 1.125), (0x40, 2.0), (0x7E, 448.0), (0xC0, -2.0),
    (0xFE, -448.0), (0x77, 240.0), (0x78, 256.0),
]


@pytest.mark.parametrize("code,value", DEFINED)
def test_defined_codes(code, value):
    v = e4m3_decode(np.array([code], dtype=np.uint8))[0]
    assert v == value and math.copysign(1.0, v) == math.copysign(1.0, value)
    assert e4m3_encode(np.array([value], dtype=np.float32))[0] == code


def test_code_table_shape():
    v = e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.isnan(v).sum() == 2 and np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)  # strictly increasing over the positive codes
    assert np.array_equal(-v[0x80:0xFF], pos)  # the sign bit mirrors
    # the distinct finite values: 127 magnitudes with both signs, +0 and -0
    assert np.isfinite(v).sum() == 254


def test_every_code_round_trips():
    c = np.arange(256, dtype=np.uint8)
    finite = c[np.isfinite(e4m3_decode(c))]
    assert np.array_equal(e4m3_encode(e4m3_decode(finite).astype(np.float32)), finite)


def _nearest_by_search(x: float) -> float:
    """The E4M3 value nearest to x by exhaustive search, ties to the even
    mantissa, magnitudes beyond 448 saturating."""
    table = e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # +0 .. 448
    a = abs(x)
    if a >= 448.0:
        return math.copysign(448.0, x)
    d = np.abs(table - a)
    best = np.flatnonzero(d == d.min())
    if best.size > 1:  # a tie: take the code with an even mantissa
        best = [b for b in best if (b & 1) == 0]
    return math.copysign(float(table[best[0]]), x)


def test_rounding_is_nearest_with_ties_to_even():
    rng = np.random.default_rng(3)
    xs = np.concatenate([
        rng.normal(0, 1, 3000), rng.normal(0, 60, 2000), rng.uniform(-2.0 ** -6, 2.0 ** -6, 1000),
        rng.uniform(400, 520, 200) * rng.choice([-1, 1], 200),
    ]).astype(np.float32)
    # exact midpoints between neighbouring codes
    tab = e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((tab[1:] + tab[:-1]) / 2).astype(np.float32)
    xs = np.concatenate([xs, mids, -mids])
    got = e4m3_decode(e4m3_encode(xs))
    for x, g in zip(xs, got):
        assert g == _nearest_by_search(float(x)), float(x)


def test_saturation_and_nan():
    c = e4m3_encode(np.array([np.inf, -np.inf, 1e30, -500.0, np.nan], dtype=np.float32))
    assert list(c[:4]) == [0x7E, 0xFE, 0x7E, 0xFE]
    assert np.isnan(e4m3_decode(c[4:]))[0]


def test_scale_divides_first():
    rng = np.random.default_rng(4)
    x = rng.normal(0, 3, 500).astype(np.float32)
    for s in (0.5, 0.0625, 3.0):
        assert np.array_equal(e4m3_encode(x, s), e4m3_encode((x / np.float32(s)).astype(np.float32)))


# --------------------------------------------------------------- FP8 pool


def _bf16(x):
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_fp8_pool_write_copy_gather():
    rng = np.random.default_rng(5)
    st = KVStore(1, 6, 4, 2, 8, "fp8_e4m3", k_scale=0.25, v_scale=2.0)
    k = _bf16(rng.normal(0, 1, (3, 2, 8)))
    v = _bf16(rng.normal(0, 1, (3, 2, 8)))
    st.reshape_and_cache(0, k, v, [5, 6, 13])
    kw = (k.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(st.K[0, 1, 1], e4m3_encode(kw[0], 0.25))
    st.copy_block(1, 4)
    assert np.array_equal(st.K[:, 4], st.K[:, 1]) and np.array_equal(st.V[:, 4], st.V[:, 1])
    kg, vg = st.gather(0, [0, 1, 0, 3], 14)
    assert np.array_equal(kg[5], e4m3_decode(st.K[0, 1, 1]) * 0.25)
    assert np.array_equal(vg[13], e4m3_decode(st.V[0, 3, 1]) * 2.0)
    # the gathered values are the quantized ones, within half a code step
    assert np.all(np.abs(kg[5] - kw[0]) <= np.abs(kw[0]) * 2.0 ** -4 + 0.25 * 2.0 ** -10)


def test_attention_over_an_fp8_pool_uses_the_dequantized_values():
    rng = np.random.default_rng(6)
    st = KVStore(1, 8, 4, 1, 16, "fp8_e4m3", k_scale=1.0, v_scale=0.5)
    k = _bf16(rng.normal(0, 1, (10, 1, 16)))
    v = _bf16(rng.normal(0, 1, (10, 1, 16)))
    table = [3, 0, 6]
    st.reshape_and_cache(0, k, v, [table[t // 4] * 4 + t % 4 for t in range(10)])
    kg, vg = st.gather(0, table, 10)
    q = rng.normal(0, 1, (2, 16))
    out = decode_attention(q, kg, vg)
    s = q @ kg[:, 0, :].T / 4.0
    w = np.exp(s - s.max(axis=1, keepdims=True))
    ref = (w / w.sum(axis=1, keepdims=True)) @ vg[:, 0, :]
    assert np.allclose(out, ref, rtol=0, atol=1e-12)
