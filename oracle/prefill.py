"""Oracle chunked-prefill attention over a paged history, float64.
TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

"KV 缓存管理" (chunked-prefill section): a prompt is split into chunks; the
queries ``Q_k`` of chunk ``k`` attend to the keys and values of every
earlier chunk, already in the paged cache, followed by the chunk's own:
``O_k = softmax(Q_k K_{<=k}^T / sqrt(d) + M_k) V_{<=k}``.  The mask ``M_k``
lets each query see the whole history and, inside the chunk, its own token
and the tokens before it.  "第 8 章 推理优化" §8.2.3 counts the pairs this
admits for a chunk of ``c`` new tokens after ``h`` cached ones:
``c * h + c (c + 1) / 2``.

* ``chunk_ranges(S, C)`` -- the token ranges of the chunks of a prompt.
* ``prefill_mask(h, c)`` -- ``[c, h + c]`` booleans: query ``i`` (position
  ``h + i``) sees key ``j`` iff ``j <= h + i``.
* ``attended_pairs(h, c)`` -- the number of admitted pairs, counted from the
  mask.
* ``prefill_attention(q, K, V)`` -- ``q [c, H_q, D_h]``, ``K, V [h + c,
  H_kv, D_h]`` (the context in logical order: history, then the chunk) ->
  ``out [c, H_q, D_h]``: every query row and head takes the softmax over the
  keys its mask row admits, with the grouped-query mapping of
  ``oracle.attention`` (query head ``x`` reads K/V head ``x // (H_q/H_kv)``).

Where the chunk's keys and values come from is left to the caller: the
pages compute them fresh and write them to the cache after the attention;
written first and read back, they are the same numbers.
"""

from __future__ import annotations

import math

import numpy as np


def chunk_ranges(s_prompt: int, c_chunk: int):
    """The chunks of a prompt of ``s_prompt`` tokens: ``K = ceil(S / C)``
    ranges, chunk ``k`` (1-based) covering tokens ``(k - 1) C`` to
    ``min(k C, S) - 1`` inclusive ("KV 缓存管理", chunked-prefill section)."""
    assert s_prompt >= 0 and c_chunk > 0
    n = -(-s_prompt // c_chunk)
    return [((k - 1) * c_chunk, min(k * c_chunk, s_prompt) - 1) for k in range(1, n + 1)]


def prefill_mask(h: int, c: int) -> np.ndarray:
    """Admitted (query, key) pairs of a chunk of ``c`` tokens after ``h``."""
    assert h >= 0 and c >= 0
    keys = np.arange(h + c)[None, :]
    pos = h + np.arange(c)[:, None]
    return keys <= pos


def attended_pairs(h: int, c: int) -> int:
    return int(prefill_mask(h, c).sum())


def prefill_attention(q, K, V, scale=None):
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    c, hq, d = q.shape
    n, hkv, d2 = K.shape
    assert d == d2 and V.shape == K.shape and n >= c
    assert hkv > 0 and hq % hkv == 0, "H_q must be a multiple of H_kv"
    h = n - c
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    group = hq // hkv
    mask = prefill_mask(h, c)
    out = np.zeros((c, hq, d), dtype=np.float64)
    for x in range(hq):
        hk = x // group
        s = (q[:, x, :] @ K[:, hk, :].T) * scale  # [c, h + c]
        s = np.where(mask, s, -np.inf)
        w = np.exp(s - s.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        out[:, x, :] = w @ V[:, hk, :]
    return out
