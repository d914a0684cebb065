"""Pins of the oracle's q8_0 codes ("第 8 章 推理优化" §8.4.2, Fig. 8-23: 32
values share one 2-byte scale and keep an 8-bit code each) against what the
layout and plain arithmetic fix, independently of the encoder's own steps:
byte counts, exact round trips of values that are already codes times a
power of two, ties to even, the fp16 rounding of the scale (checked through
Python's own half-precision packing), the zero group, sign symmetry, and
the error bound of a rounding to the nearest code."""

import struct

import numpy as np
import pytest

from oracle.kv_store import KVStore
from oracle.q8 import q8_decode, q8_encode
from oracle.sizing import GROUP32_BYTES


def f16(x: float) -> float:
    """Nearest fp16 value (Python's IEEE half packing, ties to even)."""
    return struct.unpack("<e", struct.pack("<e", x))[0]


def f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", x))[0]


def test_a_group_takes_34_bytes():
    codes, scales = q8_encode(np.ones(32, dtype=np.float32))
    assert codes.nbytes + scales.nbytes == GROUP32_BYTES["q8_0"] == 34
    assert codes.shape == (32,) and scales.shape == (1,)


def test_codes_times_a_power_of_two_round_trip_exactly():
    # x = c * 2^-7 with integer c in [-127, 127] and max |c| = 127: the scale
    # is 127 * 2^-7 / 127 = 2^-7 exactly and every code is c itself
    rng = np.random.default_rng(3)
    c = rng.integers(-127, 128, size=(5, 4, 32))
    c[..., 7] = 127 * np.where(rng.random((5, 4)) < 0.5, 1, -1)
    x = (c * 2.0 ** -7).astype(np.float32).reshape(5, 128)
    codes, scales = q8_encode(x)
    assert np.array_equal(codes.view(np.int8).reshape(5, 4, 32), c)
    assert np.all(scales.view(np.float16) == np.float16(2.0 ** -7))
    assert np.array_equal(q8_decode(codes, scales), x.astype(np.float64))


def test_ties_go_to_the_even_code():
    # scale 1 (amax 127): 2.5 -> 2, 3.5 -> 4, -2.5 -> -2, 126.5 -> 126
    x = np.zeros(32, dtype=np.float32)
    x[:5] = [127.0, 2.5, 3.5, -2.5, 126.5]
    codes, scales = q8_encode(x)
    assert scales.view(np.float16)[0] == 1.0
    assert list(codes.view(np.int8)[:5]) == [127, 2, 4, -2, 126]


def test_scale_is_the_nearest_fp16_of_amax_over_127():
    for amax in (1.0, 7.75, 0.3, 1000.0, 3.0e-3):
        x = np.zeros(32, dtype=np.float32)
        x[11] = -amax
        _, scales = q8_encode(x)
        assert scales.view(np.float16)[0] == f16(f32(f32(amax) / 127.0)), amax


def test_zero_group_and_sign_symmetry():
    codes, scales = q8_encode(np.zeros(64, dtype=np.float32))
    assert not codes.any() and not scales.any()
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 64)).astype(np.float32)
    cp, sp = q8_encode(x)
    cn, sn = q8_encode(-x)
    assert np.array_equal(sp, sn)
    assert np.array_equal(cn.view(np.int8), -cp.view(np.int8))


def test_round_trip_error_is_at_most_half_a_scale():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((200, 128)) * rng.uniform(0.01, 50, (200, 1))).astype(np.float32)
    codes, scales = q8_encode(x)
    d = np.repeat(scales.view(np.float16).astype(np.float64), 32, axis=-1)
    err = np.abs(q8_decode(codes, scales) - x.astype(np.float64))
    c = codes.view(np.int8).astype(np.int64)
    inside = np.abs(c) < 127
    # nearest code: half a scale, plus the float32 quotient's own rounding
    assert np.all(err[inside] <= d[inside] * (0.5 + 1e-6))
    # a clamped code sits where the fp16 rounding of the scale put amax
    # just past 127 scales: within half a scale plus that rounding (2^-11)
    amax = np.repeat(np.abs(x).reshape(200, 4, 32).max(-1), 32, axis=-1)
    assert np.all(err[~inside] <= d[~inside] * 0.5 + amax[~inside] * 2.0 ** -10)


@pytest.mark.parametrize("bad", [np.zeros(31, np.float32), np.zeros((2, 40), np.float32)])
def test_rows_must_hold_whole_groups(bad):
    with pytest.raises(ValueError):
        q8_encode(bad)


def test_store_writes_copies_and_gathers_q8_rows():
    st = KVStore(2, 8, 4, 2, 64, "q8_0")
    rng = np.random.default_rng(9)
    rows = (rng.standard_normal((2, 3, 2, 64)) * 3).astype(np.float32)
    bf = (rows.view(np.uint32) >> 16).astype(np.uint16)  # bf16 patterns (truncated)
    for layer in range(2):
        st.reshape_and_cache(layer, bf[layer], bf[layer], [5, 6, 9])
    st.copy_block(1, 7)  # slots 4..7 of block 1 (5 and 6 written) -> block 7
    assert np.array_equal(st.K[:, 7], st.K[:, 1]) and np.array_equal(st.Ks[:, 7], st.Ks[:, 1])
    k, v = st.gather(1, [1, 2], 6)  # block 1 holds positions 0..3, block 2 positions 4..5
    vals = (bf[1].astype(np.uint32) << 16).view(np.float32)
    ref_c, ref_s = q8_encode(vals)
    assert np.array_equal(k[1:3], q8_decode(ref_c[:2], ref_s[:2]))  # slots 5, 6
    assert np.array_equal(k[5], q8_decode(ref_c[2], ref_s[2]))       # slot 9
    assert np.array_equal(k, v)
