"""Oracle decode attention in float64.  TEST INFRASTRUCTURE ONLY.

* ``decode_attention`` -- "PagedAttention 的块表与碎片控制" §07: for the
  current query ``q_i``, ``s_t = q_i . k_t / sqrt(D_h)`` over logical
  positions ``t = 0..i`` and ``o_i = sum_t softmax(s)_t v_t``.  It runs on
  contiguous K/V (the non-paged baseline of §13); physical placement never
  enters.  Under grouped-query attention (§06) query head ``h`` reads K/V
  head ``h // (H_q / H_kv)`` (consecutive query heads share a K/V head).
* ``partial_attention`` and ``merge_partials`` -- the online-softmax
  statistics of "KV 缓存管理" (chunked-prefill section): a range of keys
  yields its running maximum ``m``, normaliser ``l = sum exp(s - m)`` and
  unnormalised output ``O = sum exp(s - m) v``; ranges merge by
  ``m = max m_i``, ``l = sum l_i exp(m_i - m)``, ``O = sum O_i exp(m_i - m)``
  and the result is ``O / l``.

An empty context (``ctx == 0``) is left open by the pages; the reading taken
here is an all-zero output.
"""

from __future__ import annotations

import math

import numpy as np


def _check(q, K, V):
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    hq, d = q.shape
    ctx, hkv, d2 = K.shape
    assert d == d2 and V.shape == K.shape
    assert hkv > 0 and hq % hkv == 0, "H_q must be a multiple of H_kv"
    return q, K, V, hq, hkv, d, ctx


def decode_attention(q, K, V, scale=None):
    """``q [H_q, D_h]``, ``K, V [ctx, H_kv, D_h]`` -> ``out [H_q, D_h]``."""
    q, K, V, hq, hkv, d, ctx = _check(q, K, V)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    group = hq // hkv
    out = np.zeros((hq, d), dtype=np.float64)
    if ctx == 0:
        return out
    for h in range(hq):
        hk = h // group
        s = (K[:, hk, :] @ q[h]) * scale
        w = np.exp(s - s.max())
        w /= w.sum()
        out[h] = w @ V[:, hk, :]
    return out


def partial_attention(q, K, V, t0, t1, scale=None):
    """Statistics ``(m [H_q], l [H_q], O [H_q, D_h])`` of keys ``t0..t1-1``.
    An empty range gives ``m = -inf``, ``l = 0``, ``O = 0``."""
    q, K, V, hq, hkv, d, ctx = _check(q, K, V)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    group = hq // hkv
    m = np.full(hq, -np.inf)
    l = np.zeros(hq)
    O = np.zeros((hq, d))
    if t1 <= t0:
        return m, l, O
    for h in range(hq):
        hk = h // group
        s = (K[t0:t1, hk, :] @ q[h]) * scale
        m[h] = s.max()
        e = np.exp(s - m[h])
        l[h] = e.sum()
        O[h] = e @ V[t0:t1, hk, :]
    return m, l, O


def merge_partials(parts):
    """Merge a list of ``(m, l, O)`` and normalise: ``out [H_q, D_h]``.
    Heads whose every range is empty get zeros."""
    ms = np.stack([p[0] for p in parts])
    ls = np.stack([p[1] for p in parts])
    Os = np.stack([p[2] for p in parts])
    m = ms.max(axis=0)
    safe_m = np.where(np.isfinite(m), m, 0.0)
    w = np.where(np.isfinite(ms), np.exp(ms - safe_m[None, :]), 0.0)
    l = (ls * w).sum(axis=0)
    O = (Os * w[:, :, None]).sum(axis=0)
    out = np.zeros_like(O)
    nz = l > 0
    out[nz] = O[nz] / l[nz, None]
    return out
