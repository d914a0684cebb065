"""The C-ABI prefix cache against the oracle (oracle/prefix_cache.py), on the
host: match lengths, slots, copy pairs, tables, counts and the cache's
statistics agree after every operation of random request streams, and both
sides' consistency checks hold.  Slots expose the allocation order, so
eviction order is compared through them."""

import numpy as np
import pytest

from oracle.block_manager import InvalidArg, NoFreeBlock
from oracle.prefix_cache import PrefixCachingBlockManager
from paged_kv_cache_65_gb300 import PagedKVCache
from paged_kv_cache_65_gb300 import _lib


def pair(N, B, salt=0, order=None):
    orc = PrefixCachingBlockManager(N, B, order, salt=salt)
    c = PagedKVCache(1, N, B, 1, 64, "f32", allocate=False, free_order=order)
    c.kv_prefix_cache_enable(salt)
    return orc, c


def same_state(orc, c, live):
    for s in live:
        t, l = c.seq_block_table([s], max(1, len(orc.tables[s])))
        assert list(t[0][: len(orc.tables[s])]) == orc.tables[s], s
        assert int(l[0]) == orc.lengths[s]
    for p in range(orc.num_blocks):
        assert c.kv_block_refcount(p) == orc.ref[p], p
    _, _, dormant, cached = orc.cache_stats()
    assert c.kv_prefix_stats() == (cached, dormant)
    assert c.kv_pool_stats()[0] == len(orc.free)
    c.kv_pool_check()
    orc.check()


def test_worked_example_through_the_abi(golden):
    ex = golden("prefix_cache_examples.json")["truncation"]
    B = ex["B"]
    orc, c = pair(64, B)
    rng = np.random.default_rng(1)
    sysp = [int(x) for x in rng.integers(0, 50000, ex["s_match"])]
    a = sysp + [int(x) for x in rng.integers(0, 50000, 30)]
    b = sysp + [int(x) for x in rng.integers(0, 50000, 20)]
    for m in (orc, c):
        assert m.seq_match_prefix(0, a) == 0 if m is c else m.match_prefix(0, a) == 0
    so, _ = orc.append_tokens(0, len(a), a)
    sc, _ = c.seq_append_tokens(0, len(a), a)
    assert list(sc) == so
    assert orc.match_prefix(1, b) == c.seq_match_prefix(1, b) == ex["usable"], ex["cite"]
    so, _ = orc.append_tokens(1, len(b) - ex["usable"], b[ex["usable"]:])
    sc, _ = c.seq_append_tokens(1, len(b) - ex["usable"], b[ex["usable"]:])
    assert list(sc) == so
    same_state(orc, c, [0, 1])


@pytest.mark.parametrize("seed", range(8))
def test_random_request_streams_match_the_oracle(seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.choice([2, 4, 8, 16]))
    N = int(rng.choice([24, 48, 96]))
    order = rng.permutation(N).astype(np.int32)
    salt = int(rng.integers(0, 2 ** 62))
    orc, c = pair(N, B, salt, order)
    vocab = int(rng.choice([3, 8, 1000]))
    bases = [[int(x) for x in rng.integers(0, vocab, 6 * B)] for _ in range(3)]
    live, nxt = [], 0
    for step in range(250):
        op = rng.random()
        if op < 0.3:
            base = bases[int(rng.integers(0, 3))]
            n = int(rng.integers(1, len(base)))
            toks = base[:n] + [int(x) for x in rng.integers(0, vocab, int(rng.integers(0, 3)))]
            sid = nxt
            nxt += 1
            mo = orc.match_prefix(sid, toks)
            mc = c.seq_match_prefix(sid, toks)
            assert mo == mc, step
            live.append(sid)
            rest = toks[mo:]
            try:
                so, po = orc.append_tokens(sid, len(rest), rest)
            except NoFreeBlock:
                so = None
            if so is None:
                with pytest.raises(Exception):
                    c.seq_append_tokens(sid, len(rest), rest)
            else:
                sc, pc = c.seq_append_tokens(sid, len(rest), rest)
                assert list(sc) == so and [tuple(x) for x in pc] == po
        elif op < 0.5 and live:
            k = int(rng.integers(1, min(4, len(live)) + 1))
            ids = [int(x) for x in rng.choice(live, k, replace=False)]
            toks = [int(x) for x in rng.integers(0, vocab, k)]
            known = rng.random() < 0.8
            try:
                so, po = orc.append_slots(ids, toks if known else None)
            except NoFreeBlock:
                so = None
            if so is None:
                with pytest.raises(Exception):
                    c.seq_append_slots(ids, toks if known else None)
            else:
                sc, pc = c.seq_append_slots(ids, toks if known else None)
                assert list(sc) == so and [tuple(x) for x in pc] == po
        elif op < 0.6 and live:
            s = int(rng.choice(live))
            orc.fork(s, nxt)
            c.seq_fork(s, nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.88 and live:
            s = int(rng.choice(live))
            orc.release(s)
            c.seq_release(s)
            live.remove(s)
        else:
            t = int(rng.integers(0, N + 1))
            assert orc.evict(t) == c.kv_prefix_evict(t)
        same_state(orc, c, live)


def test_errors():
    orc, c = pair(16, 4)
    c.seq_match_prefix(0, [1, 2, 3, 4, 5])
    with pytest.raises(Exception):
        c.seq_match_prefix(0, [1])  # exists already
    with pytest.raises(Exception):
        c.kv_prefix_cache_enable(7)  # another salt
    c.kv_prefix_cache_enable(0)  # the same salt: fine
    off = PagedKVCache(1, 8, 4, 1, 64, "f32", allocate=False)
    with pytest.raises(Exception):
        off.seq_match_prefix(0, [1, 2, 3, 4])  # cache off
