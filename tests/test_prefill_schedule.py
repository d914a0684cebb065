"""The heaviest-first chunked-prefill work order (C ABI, host only): it
holds exactly the tiles of every non-empty chunk, each tile's block count
is the number of 128-key blocks its queries read (counted here token by
token from the causal rule of the chunked-prefill section of "KV 缓存管理":
token i of a chunk after history h attends to positions 0 .. h + i), the
order is non-increasing in blocks with ties in (sequence, tile) order, and
list scheduling of the order never finishes later than the natural grid
on the pages' prefill round."""

import heapq

import numpy as np
import pytest

from paged_kv_cache_65_gb300 import PagedKVCache


def pool(H=2):
    return PagedKVCache(1, 64, 16, H, 128, "bf16", allocate=False)


def expected_items(starts, lens, G):
    T = 128 // G
    items = []
    for s in range(len(lens)):
        c = int(starts[s + 1] - starts[s])
        h = int(lens[s]) - c
        for t in range(-(-c // T)):
            toks = range(t * T, min(c, (t + 1) * T))
            last_key = max(h + i for i in toks)  # the tile's furthest position
            blocks = len({p // 128 for p in range(last_key + 1)})
            items.append((s, t, c, blocks))
    return items


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_schedule_items_blocks_and_order(seed, G):
    rng = np.random.default_rng(seed * 10 + G)
    n = int(rng.integers(1, 9))
    chunks = rng.integers(0, 700, n)
    chunks[rng.random(n) < 0.2] = 0
    hist = rng.integers(0, 3000, n)
    starts = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    lens = (hist + chunks).astype(np.int32)
    c = pool()
    got = [tuple(int(x) for x in r) for r in c.paged_prefill_schedule(starts, lens, 2 * G)]
    want = expected_items(starts, lens, G)
    assert sorted(got) == sorted(want)
    blocks = [r[3] for r in got]
    assert all(a >= b for a, b in zip(blocks, blocks[1:]))
    for a, b in zip(got, got[1:]):
        if a[3] == b[3]:
            assert (a[0], a[1]) < (b[0], b[1])


def makespan(items, n_sm=152, H=8):
    free = [0] * n_sm
    heapq.heapify(free)
    for it in items:
        for _ in range(H):
            heapq.heappush(free, heapq.heappop(free) + it[3])
    return max(free)


def test_schedule_beats_the_natural_grid_on_the_prefill_round():
    # 8 chunks of 512 tokens after histories 0 .. 7680, G = 4, 8 K/V heads
    hist = [0, 512, 1536, 2560, 3584, 4608, 5632, 7680]
    starts = np.arange(9, dtype=np.int32) * 512
    lens = np.array(hist, dtype=np.int32) + 512
    c = pool(H=8)
    sched = [tuple(r) for r in c.paged_prefill_schedule(starts, lens, 32)]
    natural = expected_items(starts, lens, 4)  # (sequence, tile) order
    total = sum(r[3] for r in natural) * 8
    assert makespan(sched) < makespan(natural)
    # within one longest item of the perfect balance (list scheduling bound)
    assert makespan(sched) <= total / 152 + max(r[3] for r in natural)


def test_schedule_errors_and_sizes():
    c = pool()
    with pytest.raises(Exception):
        c.paged_prefill_schedule([0, 10], [5], 4)  # chunk longer than its context
    with pytest.raises(Exception):
        c.paged_prefill_schedule([10, 0], [20], 4)  # negative chunk
    with pytest.raises(Exception):
        c.paged_prefill_schedule([0, 10], [20], 6)  # G = 3
    assert c.paged_prefill_schedule([0, 0, 0], [5, 9], 4).shape == (0, 4)
    from paged_kv_cache_65_gb300 import _lib

    assert _lib.lib.paged_prefill_schedule_bytes(c.handle, 3, 8, 100) == 3 * 4 * 16  # T = 32
    assert _lib.lib.paged_prefill_schedule_bytes(c.handle, 3, 7, 100) == 0


def test_staged_prefill_workspace_size():
    # an FP8 pool's staged prefill needs bfloat16 copies of K and V for
    # n_seq x max_blocks blocks of one layer (each 256-byte aligned) and the
    # copy's int32 table; a bfloat16 pool reads in place (0 bytes); invalid
    # arguments give 0
    n_seq, mb, B, H, D = 3, 7, 16, 2, 128
    f8 = PagedKVCache(2, 64, B, H, D, "fp8_e4m3", allocate=False)
    kv = n_seq * mb * B * H * D * 2
    up = lambda x: -(-x // 256) * 256  # noqa: E731
    assert f8.paged_prefill_staging_bytes(n_seq, mb) == 2 * up(kv) + up(n_seq * mb * 4)
    assert f8.paged_prefill_staging_bytes(0, mb) == 0 + 0
    assert f8.paged_prefill_staging_bytes(n_seq, 0) == 0
    assert f8.paged_prefill_staging_bytes(-1, mb) == 0
    bf = PagedKVCache(2, 64, B, H, D, "bf16", allocate=False)
    assert bf.paged_prefill_staging_bytes(n_seq, mb) == 0
