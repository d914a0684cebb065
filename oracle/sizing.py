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
* ``GROUP32_BYTES``, ``quantized_bytes``, ``bits_per_value`` -- "第 8 章 推理
  优化" §8.4.2 and Fig. 8-23: 32 BF16 values take 64 bytes; q8_0 keeps 32
  bytes of 8-bit codes plus a 2-byte scale (34), q4_0 16 bytes of 4-bit codes
  plus the scale (18); an FP8 pool with one scale per pool takes 32.  A KV
  size in BF16 scales by ``group bytes / 64``.
* ``read_saving`` -- same section: reading ``delta_bytes`` fewer bytes at an
  effective bandwidth ``beta`` saves ``delta / beta`` and the conversion
  costs ``t_convert``: ``delta / beta - t_convert``.
* ``fit_crossover`` -- the context length where two linear latency fits
  ``a + b L`` meet (the section's BF16 vs FP8 inter-token-latency fits).
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


GROUP32_BYTES = {"bf16": 64, "q8_0": 34, "q4_0": 18, "fp8_e4m3": 32}


def quantized_bytes(bf16_bytes, fmt: str) -> Fraction:
    return Fraction(bf16_bytes) * GROUP32_BYTES[fmt] / 64


def bits_per_value(fmt: str) -> Fraction:
    return Fraction(8 * GROUP32_BYTES[fmt], 32)


def read_saving(delta_bytes: float, beta: float, t_convert: float) -> float:
    return delta_bytes / beta - t_convert


def fit_crossover(a0: float, b0: float, a1: float, b1: float) -> float:
    """L where a0 + b0 L == a1 + b1 L."""
    return (a1 - a0) / (b0 - b1)
