"""Bit-exact parity of the C++ block manager (through the C ABI, host only)
with the oracle: slots, copy pairs, tables, lengths, counts, free-list order
and error codes after every operation."""

import numpy as np
import pytest

import synth
from oracle.block_manager import BlockManager, InvalidArg, NoFreeBlock, RefcountError
from paged_kv_cache_65_gb300 import KVError, PagedKVCache
from paged_kv_cache_65_gb300 import _lib

CODES = {NoFreeBlock: _lib.KV_ERR_NO_FREE_BLOCK, InvalidArg: _lib.KV_ERR_INVALID_ARG,
         RefcountError: _lib.KV_ERR_REFCOUNT}


def host_pool(n_blocks, B, order=None):
    return PagedKVCache(1, n_blocks, B, 1, 64, "f32", allocate=False, free_order=order)


def same(fn_o, fn_c):
    """Run on both; both succeed with equal results or fail with the same code."""
    try:
        ro = fn_o()
        eo = None
    except (NoFreeBlock, InvalidArg, RefcountError) as e:
        ro, eo = None, CODES[type(e)]
    try:
        rc = fn_c()
        ec = None
    except KVError as e:
        rc, ec = None, e.status
    assert eo == ec, (eo, ec)
    return ro, rc


def compare_state(bm, c, seqs):
    f, a, s = c.kv_pool_stats()
    assert (f, a, s) == bm.stats()
    c.kv_pool_check()
    bm.check()
    live = [q for q in seqs if q in bm.lengths]
    if live:
        mb = max(len(bm.tables[q]) for q in live) + 1
        tc, lc = c.seq_block_table(live, mb)
        to, lo = bm.block_table(live, mb)
        assert np.array_equal(tc, np.array(to, dtype=np.int32))
        assert np.array_equal(lc, np.array(lo, dtype=np.int32))
    for p in range(bm.num_blocks):
        assert c.kv_block_refcount(p) == bm.ref[p]


def test_worked_example_through_the_abi(golden):
    g = golden("block_table_worked_example.json")
    order = g["table"] + [g["token9_new_block"]] + [p for p in range(16) if p not in (7, 1, 3)]
    c = host_pool(16, g["block_size"], order)
    slots, pairs = c.seq_append_tokens(0, g["initial_length"])
    B = g["block_size"]
    for t, p, o in g["lookups_t_block_slot"]:
        assert slots[t] == p * B + o
    s8, _ = c.seq_append_slots([0])
    assert s8[0] == g["token8_block_slot"][0] * B + g["token8_block_slot"][1]
    s9, _ = c.seq_append_slots([0])
    assert s9[0] == g["token9_new_block"] * B
    table, lens = c.seq_block_table([0], 3)
    assert list(table[0]) == g["table_after_token9"] and lens[0] == 9


@pytest.mark.parametrize("seed", range(6))
def test_random_operation_sequences(seed):
    rng = np.random.default_rng(100 + seed)
    N, B = int(rng.integers(8, 48)), int(rng.choice([1, 2, 3, 4, 16]))
    order = rng.permutation(N)
    bm = BlockManager(N, B, order)
    c = host_pool(N, B, order)
    seqs, handles, next_id = [], [], 0
    for _ in range(400):
        op = int(rng.integers(0, 9))
        if op <= 1 or not seqs:
            s = next_id
            next_id += 1
            n = int(rng.integers(0, 3 * B + 2))
            ro, rc = same(lambda: bm.append_tokens(s, n), lambda: c.seq_append_tokens(s, n))
            if ro is not None:
                assert list(rc[0]) == ro[0]
                assert [tuple(x) for x in rc[1]] == ro[1]
                if n > 0:
                    seqs.append(s)
        elif op == 2:
            p = seqs[int(rng.integers(len(seqs)))]
            ch = next_id
            next_id += 1
            same(lambda: bm.fork(p, ch), lambda: c.seq_fork(p, ch))
            if ch in bm.lengths:
                seqs.append(ch)
        elif op == 3:
            s = seqs.pop(int(rng.integers(len(seqs))))
            same(lambda: bm.release(s), lambda: c.seq_release(s))
        elif op == 4:
            k = int(rng.integers(1, len(seqs) + 1))
            batch = [int(x) for x in rng.choice(seqs, size=k, replace=False)]
            if rng.random() < 0.2:
                batch.append(next_id)  # a brand-new sequence joins the batch
                seqs.append(next_id)
                next_id += 1
            ro, rc = same(lambda: bm.append_slots(batch), lambda: c.seq_append_slots(batch))
            if ro is not None:
                assert list(rc[0]) == ro[0]
                assert [tuple(x) for x in rc[1]] == ro[1]
            elif batch[-1] not in bm.lengths and batch[-1] in seqs:
                seqs.remove(batch[-1])
        elif op == 5:
            n = int(rng.integers(0, 4))
            ro, rc = same(lambda: bm.alloc(n), lambda: c.block_alloc(n))
            if ro is not None:
                assert list(rc) == ro
                handles.extend(ro)
        elif op == 6 and handles:
            ids = [handles.pop(int(rng.integers(len(handles))))]
            same(lambda: bm.free_blocks(ids), lambda: c.block_free(ids))
        elif op == 7 and handles:
            p = handles[int(rng.integers(len(handles)))]
            same(lambda: bm.incref([p]), lambda: c.block_fork([p]))
            handles.append(p)
        elif op == 8 and handles:
            i = int(rng.integers(len(handles)))
            ro, rc = same(lambda: bm.cow(handles[i]), lambda: c.block_cow(handles[i]))
            if ro is not None:
                assert rc == ro
                handles[i] = ro
        compare_state(bm, c, seqs)


def test_error_codes_match():
    bm, c = BlockManager(4, 2), host_pool(4, 2)
    same(lambda: bm.release(5), lambda: c.seq_release(5))
    same(lambda: bm.free_blocks([0]), lambda: c.block_free([0]))
    same(lambda: bm.incref([1]), lambda: c.block_fork([1]))
    same(lambda: bm.free_blocks([9]), lambda: c.block_free([9]))
    same(lambda: bm.append_tokens(0, 9), lambda: c.seq_append_tokens(0, 9))
    same(lambda: bm.append_slots([1, 1]), lambda: c.seq_append_slots([1, 1]))
    same(lambda: bm.fork(3, 4), lambda: c.seq_fork(3, 4))
    compare_state(bm, c, [])


@pytest.mark.parametrize("name", ["tiny", "qwen_2k", "shared_8k", "gqa70b_32k"])
def test_workload_builds_and_steps_match(name):
    wl = synth.workload(name)
    bm = BlockManager(wl.n_blocks, wl.block_size, wl.free_order)
    c = host_pool(wl.n_blocks, wl.block_size, wl.free_order)
    for op in wl.build_ops:
        if op[0] == "append":
            ro, rc = same(lambda: bm.append_tokens(op[1], op[2]),
                          lambda: c.seq_append_tokens(op[1], op[2]))
            assert np.array_equal(rc[0], np.array(ro[0], dtype=np.int64))
        elif op[0] == "fork":
            same(lambda: bm.fork(op[1], op[2]), lambda: c.seq_fork(op[1], op[2]))
        else:
            same(lambda: bm.release(op[1]), lambda: c.seq_release(op[1]))
    n_cow_first = None
    for step in range(3):
        ro, rc = same(lambda: bm.append_slots(wl.decode_seqs),
                      lambda: c.seq_append_slots(wl.decode_seqs))
        assert np.array_equal(rc[0], np.array(ro[0], dtype=np.int64))
        assert [tuple(x) for x in rc[1]] == ro[1]
        if n_cow_first is None:
            n_cow_first = len(ro[1])
    compare_state(bm, c, wl.decode_seqs)
    if name == "gqa70b_32k":
        assert n_cow_first == 48  # every branch copies the shared partial tail
    if name == "shared_8k":
        assert bm.ref[bm.tables[0][0]] == 16
