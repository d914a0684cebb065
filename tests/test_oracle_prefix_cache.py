"""Pins of the prefix-cache oracle (oracle/prefix_cache.py): the pages'
block-aligned truncation example, exact prefix identity (a token or salt
difference ends the match), leaf-first LRU eviction with cascading parents,
pinned nodes, and conservation over random operation sequences."""

import numpy as np
import pytest

from oracle.block_manager import NoFreeBlock
from oracle.prefix_cache import PrefixCachingBlockManager


def prompt(seed, n, vocab=50000):
    return [int(x) for x in np.random.default_rng(seed).integers(0, vocab, n)]


def test_block_aligned_truncation_of_the_worked_example(golden):
    ex = golden("prefix_cache_examples.json")["truncation"]
    B = ex["B"]
    m = PrefixCachingBlockManager(64, B)
    sys_prompt = prompt(1, ex["s_match"])
    # request A prefills the 100-token system prompt plus its own question
    m.match_prefix(0, sys_prompt + prompt(2, 30))
    m.append_tokens(0, 130, sys_prompt + prompt(2, 30))
    # request B shares exactly the 100 tokens, then diverges
    toks_b = sys_prompt + prompt(3, 20)
    got = m.match_prefix(1, toks_b)
    assert got == ex["usable"] == ex["full_blocks"] * B, ex["cite"]
    assert len(toks_b[:ex["s_match"]]) - got == ex["tail"]
    assert m.tables[1] == m.tables[0][: ex["full_blocks"]]
    # the 4-token tail and the suffix are new slots in a private block
    slots, cows = m.append_tokens(1, len(toks_b) - got, toks_b[got:])
    assert not cows and slots[0] // B not in m.tables[0]
    m.check()


def test_chunk_arithmetic_of_the_routing_example(golden):
    ex = golden("prefix_cache_examples.json")["chunking"]
    assert ex["S"] // ex["chunk"] * ex["chunk"] == ex["S"]
    assert ex["cached"] / ex["S"] == ex["hit"]
    assert ex["cached"] // ex["chunk"] == ex["skipped_chunks"]
    assert ex["S"] - ex["cached"] == ex["suffix"], ex["cite"]


def test_match_stops_at_the_first_differing_block():
    B = 8
    m = PrefixCachingBlockManager(32, B)
    a = prompt(4, 40)
    m.match_prefix(0, a)
    m.append_tokens(0, 40, a)
    for diff_at, want in [(0, 0), (7, 0), (8, 8), (23, 16), (24, 24), (39, 32)]:
        b = list(a)
        b[diff_at] += 1
        sid = 100 + diff_at
        assert m.match_prefix(sid, b) == want, diff_at
        m.release(sid)
    # a shorter prompt matches only its whole blocks
    assert m.match_prefix(200, a[:21]) == 16
    m.check()


def test_salt_separates_caches():
    a = prompt(5, 32)
    m = PrefixCachingBlockManager(16, 8, salt=7)
    m.match_prefix(0, a)
    m.append_tokens(0, 32, a)
    other = PrefixCachingBlockManager(16, 8, salt=8)
    other.match_prefix(0, a)
    other.append_tokens(0, 32, a)
    assert m.match_prefix(1, a) == 32
    # identical tokens under another salt: a different key, never matched
    assert other.index and not (set(other.index) & set(m.index))


def test_unknown_tokens_are_never_published():
    m = PrefixCachingBlockManager(16, 4)
    m.append_tokens(0, 12)  # no token ids
    assert m.cache_stats()[3] == 0
    m.append_tokens(1, 8, prompt(6, 8))
    assert m.cache_stats()[3] == 2


def test_leaf_first_lru_eviction_with_cascade():
    B = 4
    m = PrefixCachingBlockManager(8, B)
    trunk = prompt(7, 8)                        # two blocks
    a = trunk + prompt(8, 4)                    # trunk + leaf a
    b = trunk + prompt(9, 4)                    # trunk + leaf b
    m.match_prefix(0, a)
    m.append_tokens(0, 12, a)
    assert m.match_prefix(1, b) == 8
    m.append_tokens(1, 4, b[8:])
    t0, t1 = m.tables[0], m.tables[1]
    assert t0[:2] == t1[:2] and t0[2] != t1[2]
    m.release(1)   # leaf b dormant (trunk still held by 0)
    m.release(0)   # trunk and leaf a dormant, a touched after b
    assert m.cache_stats() == (4, 0, 4, 4)
    order = []
    while m.evict(len(m.free) + 1):
        order.append(m.free[-1])
    # leaves first, least recently used first, then the trunk upward
    assert order == [t1[2], t0[2], t0[1], t0[0]]
    m.check()


def test_pinned_blocks_are_never_evicted_and_allocation_evicts_on_demand():
    B = 4
    m = PrefixCachingBlockManager(4, B)
    a = prompt(10, 8)
    m.match_prefix(0, a)
    m.append_tokens(0, 8, a)       # 2 cached blocks, pinned by seq 0
    m.append_tokens(1, 8, prompt(11, 8))  # 2 more cached, pinned by seq 1
    with pytest.raises(NoFreeBlock):
        m.append_tokens(2, 1)       # nothing free, nothing dormant
    m.check()
    m.release(1)                    # two dormant leaves ... one leaf, one parent
    slots, _ = m.append_tokens(2, 1)  # evicts seq 1's leaf (block 2 of its chain)
    assert m.cache_stats()[2] == 1
    m.check()


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_keep_conservation(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.choice([2, 4, 8]))
    m = PrefixCachingBlockManager(48, B, salt=int(rng.integers(0, 1000)))
    bases = [prompt(seed * 10 + i, 40, vocab=6) for i in range(3)]
    live, nxt = [], 0
    for _ in range(200):
        op = rng.random()
        try:
            if op < 0.35:
                base = bases[int(rng.integers(0, 3))]
                n = int(rng.integers(1, 40))
                toks = base[:n]
                sid = nxt
                got = m.match_prefix(sid, toks)
                assert got % B == 0 and got <= n
                live.append(sid)
                nxt += 1
                m.append_tokens(sid, n - got, toks[got:])
            elif op < 0.55 and live:
                s = int(rng.choice(live))
                m.append_slots([s], [int(rng.integers(0, 6))])
            elif op < 0.65 and live:
                s = int(rng.choice(live))
                m.fork(s, nxt)
                live.append(nxt)
                nxt += 1
            elif op < 0.9 and live:
                s = int(rng.choice(live))
                m.release(s)
                live.remove(s)
            else:
                m.evict(int(rng.integers(0, 48)))
        except NoFreeBlock:
            pass
        m.check()
