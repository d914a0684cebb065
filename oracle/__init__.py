"""CPU oracle for decode attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path (``paged_kv_cache_65_gb300``) and imports nothing
from it; the only module both sides use is ``synth`` (seeded input
generators, which hold none of the method's arithmetic).

Everything here is written to be checked by eye against the pages it
follows, not to be fast:

* ``block_manager`` -- the teaching ``BlockManager`` of "PagedAttention 的块表
  与碎片控制" §05 (FIFO free list, ``append_slot``, ``release``), extended
  with the reference counts, ``fork`` and copy-on-write of "KV 缓存管理"
  (section "通过写时复制分支实现零复制审慎推理") and the atomic
  reserve-before-launch rule of "PagedAttention 的块表与碎片控制" §10.
* ``kv_store`` -- the K/V pools ``[N_layers, N_blocks, B, H_kv, D_h]`` of
  "PagedAttention 的块表与碎片控制" §06, written slot by slot, copied block
  by block, and gathered back into contiguous per-sequence arrays.
* ``attention`` -- textbook decode attention, "PagedAttention 的块表与碎片
  控制" §07, in float64 on contiguous K/V, plus the per-range partial and the
  online-softmax merge rule of "KV 缓存管理" (chunked-prefill section).
* ``sizing`` -- the closed-form sizing and waste formulas (Eq. 1, M_block,
  ceil(S/B), tail waste) used to pin the manager, and the byte arithmetic of
  narrower KV formats ("第 8 章 推理优化" §8.4.2).
* ``fp8`` -- FP8 E4M3 codes for a quantized KV pool (one scale per pool for
  K and for V), written from the format's definition; ``kv_store`` holds
  such pools.
* ``q8`` -- q8_0 codes (one fp16 scale per group of 32 values), the
  plainest rounding rule the pages' byte layout supports; ``kv_store`` holds
  such pools.
* ``q4`` -- q4_0 codes (4-bit, one fp16 scale per group of 32 values), the
  q8_0 rule with 7 in place of 127 and a stated nibble order; a codec only
  (no pool holds them).
* ``prefill`` -- chunked-prefill attention over a paged history.

Pins: every function here is checked by ``tests/test_oracle_*.py`` against
values the pages print (``tests/golden/``), closed forms, brute force or
invariants.  No function is "parity unpinned".
"""
