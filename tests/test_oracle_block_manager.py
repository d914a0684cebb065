"""Pins of ``oracle.block_manager`` and ``oracle.kv_store``.

Each test ties the oracle to a value the pages print, or to a property the
pages state (bounded waste, no aliasing, isolation after copy-on-write,
conservation), so that a plausible slip (LIFO instead of FIFO, a missing
copy-on-write, a release that forgets to return a block, an off-by-one in
``t // B`` / ``t % B``) fails one of them.
"""

import numpy as np
import pytest

from oracle import sizing
from oracle.block_manager import BlockManager, InvalidArg, NoFreeBlock, RefcountError
from oracle.kv_store import KVStore


def test_worked_block_table_example(golden):
    g = golden("block_table_worked_example.json")
    B = g["block_size"]
    # free list ordered so that the first two pops are 7 and 1 and the next is 3
    order = g["table"] + [g["token9_new_block"]] + [p for p in range(16) if p not in (7, 1, 3)]
    bm = BlockManager(16, B, order)
    got = [bm.append_slot("A")[:2] for _ in range(g["initial_length"])]
    assert bm.tables["A"] == g["table"]
    for t, p, o in g["lookups_t_block_slot"]:
        assert got[t] == (p, o)
    assert bm.append_slot("A")[:2] == tuple(g["token8_block_slot"])
    p, o, cow = bm.append_slot("A")
    assert (p, o, cow) == (g["token9_new_block"], 0, None)
    assert bm.tables["A"] == g["table_after_token9"]
    bm.check()


def test_free_list_is_fifo():
    # §05: allocation pops the head of the deque, release appends at the tail
    bm = BlockManager(4, 2)
    bm.append_slot("A")
    bm.append_slot("B")
    bm.release("A")
    assert list(bm.free) == [2, 3, 0]
    bm.append_slot("C")
    assert bm.tables["C"] == [2]
    bm.check()


def test_block_size_two_lengths_one_to_five():
    # §13: block size 2 forces frequent boundary crossings; lengths 1..5
    for n in range(1, 6):
        bm = BlockManager(8, 2, [5, 3, 7, 0, 1, 2, 4, 6])
        slots = [bm.append_slot("A") for _ in range(n)]
        assert len(bm.tables["A"]) == sizing.blocks_for(n, 2)
        for t, (p, o, _) in enumerate(slots):
            assert p == bm.tables["A"][t // 2] and o == t % 2
        assert len(bm.tables["A"]) * 2 - n == sizing.tail_waste(n, 2) <= 1
        bm.check()


def test_interleaved_sentinels_never_alias():
    # §13: interleave A, A, B, A, B, ... and write a unique (request, position)
    # sentinel into every slot; every read-back must return its own sentinel
    rng = np.random.default_rng(7)
    B, N = 2, 32
    bm = BlockManager(N, B, rng.permutation(N))
    st = KVStore(1, N, B, 1, 2, "f32")
    pattern = ["A", "A", "B", "A", "B", "C", "B", "A", "C", "C", "A", "B"] * 3
    pos = {}
    for r in pattern:
        p, o, cow = bm.append_slot(r)
        assert cow is None
        t = pos.get(r, 0)
        pos[r] = t + 1
        rid = "ABC".index(r)
        st.write_slot(0, p * B + o, [[rid, t]], [[-rid, -t]])
    for r, n in pos.items():
        k, v = st.gather(0, bm.tables[r], n)
        rid = "ABC".index(r)
        assert (k[:, 0, 0] == rid).all() and (k[:, 0, 1] == np.arange(n)).all()
        assert (v[:, 0, 0] == -rid).all() and (v[:, 0, 1] == -np.arange(n)).all()
    bm.check()


def test_tail_waste_at_most_b_minus_1():
    rng = np.random.default_rng(3)
    for B in (1, 2, 4, 5, 16):
        bm = BlockManager(4096, B)
        lens = rng.integers(1, 200, size=12)
        for s, n in enumerate(lens):
            bm.append_tokens(s, int(n))
        for s, n in enumerate(lens):
            waste = len(bm.tables[s]) * B - n
            assert 0 <= waste <= B - 1
            assert waste == sizing.tail_waste(int(n), B)
        bm.check()


def test_paging_example_with_shared_prefix(golden):
    # "第 8 章 推理优化" §8.3.1: lengths 9, 13, 5, 15 at p = 4 allocate 52 slots,
    # and 44 once A and B share their first 8 tokens (two full blocks)
    g = golden("sizing_examples.json")["paging_example"]
    B = g["block_size"]
    bm = BlockManager(64, B)
    for s, n in enumerate(g["lengths"]):
        bm.append_tokens(s, n)
    assert bm.stats()[1] * B == g["paged_total"]
    bm = BlockManager(64, B)
    bm.append_tokens("A", g["shared_prefix_tokens_ab"])
    bm.fork("A", "B")
    bm.append_tokens("A", g["lengths"][0] - 8)
    bm.append_tokens("B", g["lengths"][1] - 8)
    bm.append_tokens("C", g["lengths"][2])
    bm.append_tokens("D", g["lengths"][3])
    assert bm.tables["A"][:2] == bm.tables["B"][:2]
    assert bm.stats()[1] * B == g["paged_total_shared"]
    bm.check()


def test_branch_sharing_counts(golden):
    # "第 8 章 推理优化" §8.3.2: 4 branches x (95 shared + 9 private) blocks
    g = golden("sizing_examples.json")["branch_sharing"]
    B = 16
    bm = BlockManager(1024, B)
    bm.append_tokens("p", g["shared_blocks"] * B)
    for i in range(g["branches"]):
        bm.fork("p", i)
    bm.release("p")
    for i in range(g["branches"]):
        bm.append_tokens(i, g["private_blocks"] * B)
    refs = sum(len(bm.tables[i]) for i in range(g["branches"]))
    assert refs == g["references"]
    assert bm.stats()[1] == g["physical_blocks"]
    bm.check()


def test_shared_prefix_batch_capacity(golden):
    # "第 8 章 推理优化" §8.3.2: 16 requests sharing 6144 tokens need 6048 MiB
    g = golden("sizing_examples.json")["shared_prefix_batch"]
    B, m = g["block_size"], g["m_token"]
    bm = BlockManager(8192, B)
    bm.append_tokens("p", g["prefix_tokens"])
    assert bm.stats()[1] * B * m == g["prefix_mib"] << 20
    for i in range(g["requests"]):
        bm.fork("p", i)
    bm.release("p")
    for i in range(g["requests"]):
        bm.append_tokens(i, g["private_tokens"])
    assert bm.stats()[1] * B * m == g["total_mib"] << 20
    assert len(bm.tables[0][g["prefix_tokens"] // B:]) * B * m == g["private_mib"] << 20
    bm.check()


def test_fork_then_cow_isolates_branches():
    # "第 8 章 推理优化" §8.3.2 / Fig. 8-15: a 4-slot tail holding a, b, c is
    # shared; the branches append x and y; each needs its own tail while the
    # full blocks before it stay shared and untouched
    B = 4
    bm = BlockManager(16, B, list(range(15, -1, -1)))
    st = KVStore(1, 16, B, 1, 1, "f32")

    def put(seq, val):
        p, o, cow = bm.append_slot(seq)
        if cow is not None:
            st.copy_block(*cow)
        st.write_slot(0, p * B + o, [[val]], [[val]])
        return cow

    for i in range(7):  # one full block + a, b, c
        put("A", 100 + i)
    bm.fork("A", "B")
    before = (list(bm.tables["A"]), st.K.copy())
    assert bm.tables["A"] == bm.tables["B"]
    assert [bm.ref[p] for p in bm.tables["A"]] == [2, 2]
    cow_a = put("A", 1.5)  # x: A is the first writer into the shared tail: copies
    cow_b = put("B", 2.5)  # y: B is now the tail's only holder: writes in place
    assert cow_a == (before[0][1], bm.tables["A"][1]) and cow_b is None
    assert bm.tables["A"][0] == bm.tables["B"][0]          # full block still shared
    assert bm.tables["A"][1] != bm.tables["B"][1]          # tails are private
    ka, _ = st.gather(0, bm.tables["A"], 8)
    kb, _ = st.gather(0, bm.tables["B"], 8)
    assert list(ka[:, 0, 0]) == [100, 101, 102, 103, 104, 105, 106, 1.5]
    assert list(kb[:, 0, 0]) == [100, 101, 102, 103, 104, 105, 106, 2.5]
    # the shared full block is bit-identical before and after divergence
    p0 = bm.tables["A"][0]
    assert np.array_equal(st.K[:, p0], before[1][:, p0])
    bm.check()


def test_release_returns_blocks_in_table_order():
    # "KV 缓存管理", release_sequence_blocks: walk the table, return blocks
    # whose count reaches zero to the free list tail
    bm = BlockManager(8, 2)
    bm.append_tokens("A", 6)  # blocks 0, 1, 2
    bm.fork("A", "B")
    bm.append_tokens("B", 2)  # block 3
    bm.release("A")
    assert list(bm.free) == [4, 5, 6, 7]
    bm.release("B")
    assert list(bm.free) == [4, 5, 6, 7, 0, 1, 2, 3]
    bm.check()


def test_batch_append_is_atomic():
    # "PagedAttention 的块表与碎片控制" §10: reserve everything or nothing
    bm = BlockManager(3, 2)
    bm.append_tokens(0, 2)
    bm.append_tokens(1, 2)
    snap = (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()}, dict(bm.lengths))
    with pytest.raises(NoFreeBlock):
        bm.append_slots([0, 1])  # needs two new blocks, only one is free
    assert (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()}, dict(bm.lengths)) == snap
    slots, cows = bm.append_slots([0])
    assert slots == [2 * 2 + 0] and cows == []
    with pytest.raises(InvalidArg):
        bm.append_slots([1, 1])
    bm.check()


def test_block_level_handles_and_errors():
    bm = BlockManager(4, 2)
    ids = bm.alloc(2)
    assert ids == [0, 1]
    with pytest.raises(NoFreeBlock):
        bm.alloc(3)
    assert bm.stats() == (2, 2, 0)
    bm.incref([0])
    assert bm.stats() == (2, 2, 1)
    new = bm.cow(0)
    assert new == 2 and bm.ref[0] == 1 and bm.ref[2] == 1
    assert bm.cow(1) == 1  # not shared: write in place
    bm.free_blocks([0, 1, 2])
    assert bm.stats() == (4, 0, 0)
    assert list(bm.free) == [3, 0, 1, 2]
    with pytest.raises(RefcountError):
        bm.free_blocks([0])  # double free
    with pytest.raises(RefcountError):
        bm.incref([0])  # sharing a free block
    with pytest.raises(InvalidArg):
        bm.free_blocks([9])
    bm.check()


def test_error_paths_conserve_state():
    # §13: no free block, cancellation and exceptions must conserve the
    # reference counts and the free list
    rng = np.random.default_rng(11)
    bm = BlockManager(40, 3, rng.permutation(40))
    live = []
    next_id = 0
    for step in range(600):
        op = rng.integers(0, 5)
        try:
            if op == 0 or not live:
                s = next_id
                next_id += 1
                bm.append_tokens(s, int(rng.integers(1, 12)))
                live.append(s)
            elif op == 1:
                s = live[rng.integers(len(live))]
                c = next_id
                next_id += 1
                bm.fork(s, c)
                live.append(c)
            elif op == 2:
                s = live.pop(rng.integers(len(live)))
                bm.release(s)
            else:
                k = int(rng.integers(1, len(live) + 1))
                batch = list(rng.choice(live, size=k, replace=False))
                bm.append_slots(batch)
        except NoFreeBlock:
            pass
        bm.check()
    for s in live:
        bm.release(s)
    assert bm.stats() == (40, 0, 0)
    bm.check()


def test_runner_places_each_sequence_values_in_logical_order():
    # the oracle run of the tiny recipe: every sequence's gather equals the
    # values its append ops drew, in order, and the step's own token is last
    import synth
    from oracle.runner import OracleRun

    wl = synth.workload("tiny")
    run = OracleRun(wl)
    per_seq = {s: ([], []) for s in wl.decode_seqs}
    for op in wl.build_ops:
        _, s, n, vs = op
        k, v = wl.append_values(vs, n)
        per_seq[s][0].append(k[0])
        per_seq[s][1].append(v[0])
    slots, cows, q, outs = run.step(0)
    assert cows == []
    _, k_new, v_new = wl.step_values(0)
    for i, s in enumerate(wl.decode_seqs):
        K, V = run.st.gather_raw(0, run.bm.tables[s], run.bm.lengths[s])
        want_k = np.concatenate(per_seq[s][0] + [k_new[0, i:i + 1]])
        want_v = np.concatenate(per_seq[s][1] + [v_new[0, i:i + 1]])
        assert np.array_equal(K, want_k) and np.array_equal(V, want_v)
    assert [run.bm.lengths[s] for s in wl.decode_seqs] == [7, 13, 1, 16]
    run.bm.check()
