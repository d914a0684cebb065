"""Pins of the oracle's q4_0 codes ("第 8 章 推理优化" §8.4.2, Fig. 8-23: 32
values share one 2-byte scale and keep a 4-bit code each) against what the
layout and plain arithmetic fix, independently of the encoder's own steps:
the 18-byte group, a hand-packed byte pattern for the nibble order, exact
round trips of values that are already codes times a power of two, ties to
even, the fp16 rounding of the scale (Python's own half-precision packing),
the zero group, sign symmetry, and the half-scale error bound."""

import struct

import numpy as np
import pytest

from oracle.q4 import q4_codes, q4_decode, q4_encode, q4_pack, q4_unpack
from oracle.sizing import GROUP32_BYTES


def f16(x: float) -> float:
    """Nearest fp16 value (Python's IEEE half packing, ties to even)."""
    return struct.unpack("<e", struct.pack("<e", x))[0]


def f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", x))[0]


def test_a_group_takes_18_bytes():
    packed, scales = q4_encode(np.ones(32, dtype=np.float32))
    assert packed.nbytes + scales.nbytes == GROUP32_BYTES["q4_0"] == 18
    assert packed.shape == (16,) and scales.shape == (1,)


def test_nibble_order_by_hand():
    # scale 1 (amax 7): codes 7, -7, 1, 0, -1, 3 ... stored as c + 8, the
    # even-indexed value in the low nibble
    x = np.zeros(32, dtype=np.float32)
    x[:6] = [7.0, -7.0, 1.0, 0.0, -1.0, 3.0]
    packed, scales = q4_encode(x)
    assert scales.view(np.float16)[0] == 1.0
    assert list(packed[:3]) == [(15 | (1 << 4)), (9 | (8 << 4)), (7 | (11 << 4))]
    assert all(b == (8 | (8 << 4)) for b in packed[3:])


def test_pack_and_unpack_are_inverse():
    rng = np.random.default_rng(1)
    c = rng.integers(-7, 8, size=(3, 64)).astype(np.int8)
    assert np.array_equal(q4_unpack(q4_pack(c)), c)


def test_codes_times_a_power_of_two_round_trip_exactly():
    # x = c * 2^-3 with integer c in [-7, 7] and max |c| = 7: the scale is
    # 7 * 2^-3 / 7 = 2^-3 exactly and every code is c itself
    rng = np.random.default_rng(3)
    c = rng.integers(-7, 8, size=(5, 4, 32))
    c[..., 5] = 7 * np.where(rng.random((5, 4)) < 0.5, 1, -1)
    x = (c * 2.0 ** -3).astype(np.float32).reshape(5, 128)
    codes, scales = q4_codes(x)
    assert np.array_equal(codes.reshape(5, 4, 32), c)
    assert np.all(scales.view(np.float16) == np.float16(2.0 ** -3))
    packed, scales = q4_encode(x)
    assert np.array_equal(q4_decode(packed, scales), x.astype(np.float64))


def test_ties_go_to_the_even_code():
    # scale 1 (amax 7): 2.5 -> 2, 3.5 -> 4, -2.5 -> -2, 6.5 -> 6
    x = np.zeros(32, dtype=np.float32)
    x[:5] = [7.0, 2.5, 3.5, -2.5, 6.5]
    codes, scales = q4_codes(x)
    assert scales.view(np.float16)[0] == 1.0
    assert list(codes[:5]) == [7, 2, 4, -2, 6]


def test_scale_is_the_nearest_fp16_of_amax_over_7():
    for amax in (1.0, 7.75, 0.3, 1000.0, 3.0e-3):
        x = np.zeros(32, dtype=np.float32)
        x[20] = -amax
        _, scales = q4_codes(x)
        assert scales.view(np.float16)[0] == f16(f32(f32(amax) / 7.0)), amax


def test_zero_group_and_sign_symmetry():
    codes, scales = q4_codes(np.zeros(64, dtype=np.float32))
    assert not codes.any() and not scales.any()
    packed, _ = q4_encode(np.zeros(64, dtype=np.float32))
    assert np.all(packed == 0x88)  # code 0 is the nibble 8
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 64)).astype(np.float32)
    cp, sp = q4_codes(x)
    cn, sn = q4_codes(-x)
    assert np.array_equal(sp, sn) and np.array_equal(cn, -cp)


def test_round_trip_error_is_at_most_half_a_scale():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((200, 128)) * rng.uniform(0.01, 50, (200, 1))).astype(np.float32)
    packed, scales = q4_encode(x)
    d = np.repeat(scales.view(np.float16).astype(np.float64), 32, axis=-1)
    err = np.abs(q4_decode(packed, scales) - x.astype(np.float64))
    c = q4_unpack(packed).astype(np.int64)
    inside = np.abs(c) < 7
    assert np.all(err[inside] <= d[inside] * (0.5 + 1e-6))
    # a clamped code sits where the fp16 rounding of the scale put amax
    # just past 7 scales: within half a scale plus that rounding (2^-11)
    amax = np.repeat(np.abs(x).reshape(200, 4, 32).max(-1), 32, axis=-1)
    assert np.all(err[~inside] <= d[~inside] * 0.5 + amax[~inside] * 2.0 ** -10)


@pytest.mark.parametrize("bad", [np.zeros(31, np.float32), np.zeros((2, 40), np.float32)])
def test_rows_must_hold_whole_groups(bad):
    with pytest.raises(ValueError):
        q4_encode(bad)
