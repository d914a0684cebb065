"""Pins of ``oracle.attention`` (and of the gather in ``oracle.kv_store``).

Closed forms and special cases that the decode formula of
"PagedAttention 的块表与碎片控制" §07 fixes, an arbitrary-precision brute
force on small inputs, invariance under physical placement (§03, §07: "the
blocks are not contiguous, which changes neither positions nor the softmax
denominator"), and the online-softmax merge rule of "KV 缓存管理".
"""

import math

import numpy as np
import pytest

from oracle.attention import decode_attention, merge_partials, partial_attention
from oracle.block_manager import BlockManager
from oracle.kv_store import KVStore, to_f64


def rand(rng, *shape):
    return rng.standard_normal(shape)


def test_single_token_returns_its_value_exactly():
    rng = np.random.default_rng(0)
    q, K, V = rand(rng, 8, 64), rand(rng, 1, 2, 64), rand(rng, 1, 2, 64)
    out = decode_attention(q, K, V)
    for h in range(8):
        assert np.array_equal(out[h], V[0, h // 4])


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(1)
    K, V = rand(rng, 13, 2, 16), rand(rng, 13, 2, 16)
    out = decode_attention(np.zeros((6, 16)), K, V)
    for h in range(6):
        np.testing.assert_allclose(out[h], V[:, h // 3].mean(axis=0), rtol=0, atol=1e-14)


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    k = rand(rng, 2, 16)
    K = np.repeat(k[None], 9, axis=0)
    V = rand(rng, 9, 2, 16)
    out = decode_attention(rand(rng, 4, 16), K, V)
    for h in range(4):
        np.testing.assert_allclose(out[h], V[:, h // 2].mean(axis=0), rtol=0, atol=1e-14)


def test_constant_values_pass_through():
    rng = np.random.default_rng(3)
    v = rand(rng, 2, 8)
    V = np.repeat(v[None], 11, axis=0)
    out = decode_attention(rand(rng, 4, 8), rand(rng, 11, 2, 8), V)
    for h in range(4):
        np.testing.assert_allclose(out[h], v[h // 2], rtol=0, atol=1e-14)


def test_two_token_logistic_closed_form_pins_scale_and_direction():
    # two keys: weights are sigmoid(s0 - s1) and 1 - that, s_t = q.k_t / sqrt(D)
    D = 16
    q = np.zeros((1, D))
    q[0, 0] = 3.0
    K = np.zeros((2, 1, D))
    K[0, 0, 0] = 1.0  # s0 = 3 / 4
    V = np.zeros((2, 1, D))
    V[0, 0, 1] = 1.0
    V[1, 0, 2] = 1.0
    w0 = 1.0 / (1.0 + math.exp(-(3.0 / 4.0)))
    out = decode_attention(q, K, V)
    assert abs(out[0, 1] - w0) < 1e-15 and abs(out[0, 2] - (1 - w0)) < 1e-15


def test_gqa_head_mapping():
    # query head h reads K/V head h // (H_q / H_kv): give every K/V head a
    # distinct constant value row
    H_kv, G, D = 4, 3, 8
    V = np.zeros((5, H_kv, D))
    for hk in range(H_kv):
        V[:, hk, :] = hk + 1
    out = decode_attention(np.ones((H_kv * G, D)), np.ones((5, H_kv, D)), V)
    for h in range(H_kv * G):
        np.testing.assert_allclose(out[h], h // G + 1, rtol=0, atol=1e-14)


def test_against_arbitrary_precision_brute_force():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    rng = np.random.default_rng(4)
    Hq, Hkv, D = 4, 2, 8
    for ctx in (1, 2, 5, 16):
        q, K, V = rand(rng, Hq, D), rand(rng, ctx, Hkv, D), rand(rng, ctx, Hkv, D)
        out = decode_attention(q, K, V)
        for h in range(Hq):
            hk = h // (Hq // Hkv)
            s = [mp.fsum(mp.mpf(q[h, d]) * mp.mpf(K[t, hk, d]) for d in range(D)) / mp.sqrt(D)
                 for t in range(ctx)]
            e = [mp.exp(x) for x in s]
            z = mp.fsum(e)
            for d in range(D):
                ref = mp.fsum(e[t] * mp.mpf(V[t, hk, d]) for t in range(ctx)) / z
                assert abs(float(ref) - out[h, d]) < 1e-13


def test_empty_context_is_zero():
    out = decode_attention(np.ones((4, 8)), np.zeros((0, 2, 8)), np.zeros((0, 2, 8)))
    assert out.shape == (4, 8) and not out.any()


def test_merge_over_every_split_equals_unsplit():
    rng = np.random.default_rng(5)
    Hq, Hkv, D, ctx = 4, 2, 8, 11
    q, K, V = rand(rng, Hq, D), rand(rng, ctx, Hkv, D), rand(rng, ctx, Hkv, D)
    ref = decode_attention(q, K, V)
    for a in range(ctx + 1):
        for b in range(a, ctx + 1):
            parts = [partial_attention(q, K, V, 0, a), partial_attention(q, K, V, a, b),
                     partial_attention(q, K, V, b, ctx)]
            np.testing.assert_allclose(merge_partials(parts), ref, rtol=0, atol=1e-13)
    # one range per token, scrambled order: the merge is order-free
    parts = [partial_attention(q, K, V, t, t + 1) for t in rng.permutation(ctx)]
    np.testing.assert_allclose(merge_partials(parts), ref, rtol=0, atol=1e-13)
    assert not merge_partials([partial_attention(q, K, V, 3, 3)]).any()


def test_partial_single_token_statistics():
    rng = np.random.default_rng(6)
    q, K, V = rand(rng, 2, 8), rand(rng, 4, 1, 8), rand(rng, 4, 1, 8)
    m, l, O = partial_attention(q, K, V, 2, 3)
    for h in range(2):
        assert m[h] == pytest.approx(K[2, 0] @ q[h] / math.sqrt(8), abs=1e-15)
        assert l[h] == 1.0 and np.array_equal(O[h], V[2, 0])


def test_placement_invariance_through_paged_store():
    # the same logical tokens placed on two different free-list orders give
    # bit-identical gathers and outputs
    rng = np.random.default_rng(8)
    B, N, H, D = 4, 64, 2, 16
    ctx = [7, 13, 1, 16]
    toks = [rand(rng, c, 2, H, D).astype(np.float32) for c in ctx]
    q = rand(rng, len(ctx), 8, D)
    outs = []
    for order in (np.arange(N), rng.permutation(N)):
        bm = BlockManager(N, B, order)
        st = KVStore(1, N, B, H, D, "f32")
        for t in range(max(ctx)):
            for s, c in enumerate(ctx):
                if t < c:
                    p, o, _ = bm.append_slot(s)
                    st.write_slot(0, p * B + o, toks[s][t, 0], toks[s][t, 1])
        res = []
        for s, c in enumerate(ctx):
            K, V = st.gather(0, bm.tables[s], c)
            assert np.array_equal(K, toks[s][:, 0].astype(np.float64))
            assert np.array_equal(V, toks[s][:, 1].astype(np.float64))
            res.append(decode_attention(q[s], K, V))
        outs.append(res)
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_bf16_widening_is_exact():
    # bf16 pattern h stands for the float32 with bits h << 16
    pats = np.array([0x0000, 0x3F80, 0xBF80, 0x4049, 0x7F7F, 0x0001, 0xC2F7], dtype=np.uint16)
    want = [0.0, 1.0, -1.0, 3.140625, 3.3895313892515355e38, 9.183549615799121e-41, -123.5]
    assert list(to_f64(pats, "bf16")) == want
