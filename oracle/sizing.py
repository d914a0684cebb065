"""Closed-form sizing and waste formulas.  TEST INFRASTRUCTURE ONLY.

* ``m_token`` -- "KV 缓存管理" Eq. 1 (also "PagedAttention 的块表与碎片控制"
  §01 and "第 8 章 推理优化" §8.1.2): ``2 * L * H_kv * d_head * b`` bytes per
  token, the 2 counting K and V.
* ``m_block`` -- "KV 缓存管理", section "PagedAttention 虚拟内存模型":
  ``2 * L * H_kv * B * d_head * b`` bytes per physical block.
* ``blocks_for`` -- same section: ``ceil(S / B)`` blocks hold ``S`` tokens.
* ``tail_waste`` -- "KV 缓存管理", section "块大小选择中的量化权衡":
  ``(B - S mod B) mod B`` unused slots in the last block; "第 8 章 推理优化"
  §8.3.1 writes the same as ``p * ceil(L / p) - L``.
* ``mean_tail_waste`` -- the expectation of ``tail_waste`` when ``S mod B`` is
  uniform on ``0..B-1``, evaluated as that average (the pages state its value
  ``(B - 1) / 2``; the tests check the two agree).
"""

from __future__ import annotations

from fractions import Fraction


def m_token(n_layers: int, n_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return 2 * n_layers * n_kv_heads * head_dim * elem_bytes


def m_block(n_layers: int, n_kv_heads: int, head_dim: int, elem_bytes: int, block_size: int) -> int:
    return 2 * n_layers * n_kv_heads * block_size * head_dim * elem_bytes


def blocks_for(tokens: int, block_size: int) -> int:
    return -(-tokens // block_size)


def tail_waste(tokens: int, block_size: int) -> int:
    return (block_size - tokens % block_size) % block_size


def paged_slots(lengths, block_size: int) -> int:
    """Slots allocated to a set of private sequences."""
    return sum(block_size * blocks_for(s, block_size) for s in lengths)


def mean_tail_waste(block_size: int) -> Fraction:
    return Fraction(sum(tail_waste(r, block_size) for r in range(block_size)), block_size)
