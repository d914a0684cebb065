"""Pins of the chunked-prefill oracle (oracle/prefill.py) to what the pages
print and to properties that any correct causal attention over a paged
history has."""

import math

import numpy as np
import pytest

from oracle.attention import decode_attention
from oracle.prefill import attended_pairs, chunk_ranges, prefill_attention, prefill_mask


def test_pair_counts_printed_on_the_pages(golden):
    g = golden("prefill_examples.json")
    for ex in g["attended_pairs"]:
        assert attended_pairs(ex["h"], ex["c"]) == ex["pairs"], ex["cite"]
    first = attended_pairs(0, 512)
    last = attended_pairs(7680, 512)
    assert round(last / first) == g["pairs_ratio_last_to_first"]["ratio"]


@pytest.mark.parametrize("h,c", [(0, 1), (0, 7), (5, 1), (13, 9), (100, 64)])
def test_pair_count_closed_form(h, c):
    # every query sees the whole history plus a triangle inside the chunk
    assert attended_pairs(h, c) == c * h + c * (c + 1) // 2


def test_chunk_ranges_of_the_worked_example(golden):
    ex = golden("prefill_examples.json")["chunk_ranges"][0]
    r = chunk_ranges(ex["S"], ex["C"])
    assert len(r) == ex["K"]
    first, last = r[ex["k"] - 1]
    assert (first, last) == (ex["first"], ex["last"])
    # the last query of chunk k sees every key up to its own position
    m = prefill_mask(first, last - first + 1)
    assert m[-1].sum() == ex["keys_of_last_query"]
    # ragged last chunk, and the chunks tile the prompt
    assert chunk_ranges(1000, 512) == [(0, 511), (512, 999)]
    assert chunk_ranges(0, 512) == []


def rand(rng, *shape):
    return rng.standard_normal(shape)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(0)
    q, K, V = rand(rng, 1, 4, 8), rand(rng, 1, 2, 8), rand(rng, 1, 2, 8)
    out = prefill_attention(q, K, V)
    for x in range(4):
        assert np.array_equal(out[0, x], V[0, x // 2])


def test_two_keys_logistic_closed_form():
    # one cached key and one chunk token: the second query row weighs its two
    # keys by a logistic of the scaled score difference
    rng = np.random.default_rng(1)
    d = 16
    q, K, V = rand(rng, 1, 1, d), rand(rng, 2, 1, d), rand(rng, 2, 1, d)
    out = prefill_attention(q, K, V)
    s0 = q[0, 0] @ K[0, 0] / math.sqrt(d)
    s1 = q[0, 0] @ K[1, 0] / math.sqrt(d)
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    assert np.allclose(out[0, 0], (1 - w1) * V[0, 0] + w1 * V[1, 0], atol=1e-13)


def test_identical_keys_give_the_mean_of_the_visible_values():
    rng = np.random.default_rng(2)
    h, c, d = 5, 6, 8
    K = np.repeat(rand(rng, 1, 1, d), h + c, axis=0)
    V = rand(rng, h + c, 1, d)
    q = rand(rng, c, 3, d)
    out = prefill_attention(q, K, V)
    for i in range(c):
        assert np.allclose(out[i, :], V[: h + i + 1, 0].mean(axis=0), atol=1e-12)


def test_rows_do_not_see_future_tokens():
    rng = np.random.default_rng(3)
    h, c = 7, 9
    q, K, V = rand(rng, c, 4, 16), rand(rng, h + c, 2, 16), rand(rng, h + c, 2, 16)
    base = prefill_attention(q, K, V)
    for t in range(h, h + c):
        K2, V2 = K.copy(), V.copy()
        K2[t] += 5.0
        V2[t] -= 3.0
        out = prefill_attention(q, K2, V2)
        i = t - h
        assert np.array_equal(out[:i], base[:i])   # earlier rows untouched
        assert not np.allclose(out[i], base[i])    # the token's own row sees it


def test_one_token_chunk_is_decode_attention():
    rng = np.random.default_rng(4)
    h = 20
    q, K, V = rand(rng, 1, 8, 32), rand(rng, h + 1, 2, 32), rand(rng, h + 1, 2, 32)
    assert np.allclose(prefill_attention(q, K, V)[0], decode_attention(q[0], K, V), atol=1e-13)


def test_chunking_leaves_the_outputs_unchanged():
    # "KV 缓存管理": chunked prefill is mathematically equivalent to one pass
    rng = np.random.default_rng(5)
    S, hq, hkv, d = 37, 4, 2, 16
    q, K, V = rand(rng, S, hq, d), rand(rng, S, hkv, d), rand(rng, S, hkv, d)
    whole = prefill_attention(q, K, V)
    for C in (1, 5, 16, 36):
        parts = []
        for a, b in chunk_ranges(S, C):
            parts.append(prefill_attention(q[a:b + 1], K[:b + 1], V[:b + 1]))
        assert np.allclose(np.concatenate(parts), whole, atol=1e-12), C


def test_last_row_of_a_chunk_is_decode_over_the_whole_context():
    rng = np.random.default_rng(6)
    h, c = 30, 12
    q, K, V = rand(rng, c, 8, 16), rand(rng, h + c, 2, 16), rand(rng, h + c, 2, 16)
    out = prefill_attention(q, K, V)
    assert np.allclose(out[-1], decode_attention(q[-1], K, V), atol=1e-13)
    assert np.allclose(out[3], decode_attention(q[3], K[: h + 4], V[: h + 4]), atol=1e-13)
