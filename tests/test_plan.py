"""The sharing-aware decode plan (host, through the C ABI) against the
oracle's block tables: every (sequence, K/V head) is covered by its merge
entries exactly once over [0, context), every segment reads, for each member,
the very physical blocks that member's own table names, and shared segments
carry all their members' query heads."""

import numpy as np
import pytest

import synth
from oracle.block_manager import BlockManager
from paged_kv_cache_65_gb300 import PagedKVCache
from paged_kv_cache_65_gb300.cache import parse_plan


def build_both(wl):
    bm = BlockManager(wl.n_blocks, wl.block_size, wl.free_order)
    c = PagedKVCache(1, wl.n_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim, wl.dtype,
                     allocate=False, free_order=wl.free_order)
    for op in wl.build_ops:
        if op[0] == "append":
            bm.append_tokens(op[1], op[2])
            c.seq_append_tokens(op[1], op[2])
        elif op[0] == "fork":
            bm.fork(op[1], op[2])
            c.seq_fork(op[1], op[2])
        else:
            bm.release(op[1])
            c.seq_release(op[1])
    bm.append_slots(wl.decode_seqs)
    c.seq_append_slots(wl.decode_seqs)
    return bm, c


def check_plan(bm, plan, seqs, G, min_tokens):
    B, H = plan["B"], plan["H"]
    segs, mem, eoff, ents = plan["segs"], plan["members"], plan["eoff"], plan["ents"]
    assert plan["G"] == G and plan["n_seq"] == len(seqs)
    units = [int(s["b1"] - s["b0"]) * int(s["w"]) for s in segs]
    assert plan["W"] == sum(units)
    assert list(segs["wpre"]) == list(np.cumsum([0] + units)[:-1])
    # units per block: 8 per part of the block's cost, plus the piece's fixed
    # cost (one stage of narrow blocks, two on tcgen05) spread over the
    # segment's blocks
    for s in segs:
        n = int(s["b1"] - s["b0"])
        if plan["kernel"] == 3:  # tcgen05
            base, piece = 8 * (4 if s["ncols"] <= 16 else 5), 32 * 32
        else:
            assert plan["kernel"] == 2
            base, piece = 8 * (3 if s["ncols"] <= 8 else 4 if s["ncols"] <= 16 else 5), 4 * 24
        assert s["w"] == base + (-(-piece // n) if n > 0 else 0)
    for si, s in enumerate(segs):
        assert s["ncols"] % G == 0 and 0 < s["ncols"] <= 32
        members = mem[s["mem"]:s["mem"] + s["ncols"] // G]
        assert s["rep"] == members[0]
        rep_table = bm.tables[seqs[s["rep"]]]
        for m in members:
            t = bm.tables[seqs[m]]
            # the segment's blocks are this member's own blocks, inside its context
            assert t[s["b0"]:s["b1"]] == rep_table[s["b0"]:s["b1"]]
            assert s["tok_end"] <= bm.lengths[seqs[m]]
        if len(members) > 1:
            assert s["tok_end"] == s["b1"] * B and s["b1"] * B >= min_tokens
    for i, sid in enumerate(seqs):
        L = bm.lengths[sid]
        for h in range(H):
            covered = np.zeros(L, dtype=np.int64)
            for e in ents[eoff[i * H + h]:eoff[i * H + h + 1]]:
                s = segs[e["seg"]]
                assert s["head"] == h
                members = list(mem[s["mem"]:s["mem"] + s["ncols"] // G])
                assert members.index(i) * G == e["col_base"]
                covered[s["b0"] * B:min(s["b1"] * B, s["tok_end"])] += 1
            assert (covered == 1).all(), (sid, h)


@pytest.mark.parametrize("path", [0, 3])
@pytest.mark.parametrize("name", ["tiny", "qwen_2k", "shared_8k", "gqa70b_32k", "qwen_2k_fp8",
                                  "shared_8k_fp8", "gqa70b_32k_fp8", "qwen_2k_q8"])
def test_plans_of_the_workloads(name, path):
    from paged_kv_cache_65_gb300 import _lib

    wl = synth.workload(name)
    bm, c = build_both(wl)
    c.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, path)
    G = wl.n_q_heads // wl.n_kv_heads
    mb = max(len(bm.tables[s]) for s in wl.decode_seqs)
    buf, ws = c.paged_decode_plan(wl.decode_seqs, wl.n_q_heads, mb)
    plan = parse_plan(buf)
    check_plan(bm, plan, wl.decode_seqs, G, 128)
    # the tcgen05 kernel is for bfloat16 and FP8 pools with D_h = 128 and B a
    # multiple of 8 (q8_0 pools take the warp-level pass)
    tc_shape = (wl.dtype in ("bf16", "fp8_e4m3") and wl.head_dim == 128
                and wl.block_size % 8 == 0)
    # automatic: tcgen05 when segments wider than 16 columns hold half of the blocks
    wide = sum(int(s["b1"] - s["b0"]) for s in plan["segs"] if s["ncols"] > 16)
    total = sum(int(s["b1"] - s["b0"]) for s in plan["segs"])
    auto_tc = 2 * wide >= total
    assert plan["kernel"] == (3 if tc_shape and (path == 3 or auto_tc) else 2)
    base = name.replace("_fp8", "").replace("_q8", "")
    if base == "gqa70b_32k":
        assert auto_tc
    assert ws > 0
    shared = [s for s in plan["segs"] if s["ncols"] > G]
    if base == "gqa70b_32k":
        # 12 parents x 4 branches: one shared segment per parent and K/V head
        assert len(shared) == 12 * 8 and all(s["ncols"] == 32 for s in shared)
        assert all(s["b1"] == 2048 for s in shared)
    elif base == "shared_8k":
        # 16 sharers of 384 blocks at G = 4: two sub-groups of 8 per K/V head
        assert len(shared) == 2 * 8 and all(s["b1"] == 384 for s in shared)
    else:
        assert not shared


@pytest.mark.parametrize("seed", range(5))
def test_plans_of_random_fork_trees(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.choice([8, 16]))
    H, G = 2, int(rng.choice([1, 2, 4, 8]))
    ops, live, nxt = [], [], 0
    for _ in range(8):
        ops.append(("append", nxt, int(rng.integers(1, 300)), nxt))
        live.append(nxt)
        nxt += 1
    for _ in range(30):
        p = int(rng.choice(live))
        if rng.random() < 0.5:
            ops.append(("fork", p, nxt))
            live.append(nxt)
            nxt += 1
        else:
            ops.append(("append", p, int(rng.integers(1, 40)), nxt))
    wl = synth.Workload("forks", 1, 4096, B, H * G, H, 128, "bf16", seed, None, ops, live)
    bm, c = build_both(wl)
    mb = max(len(bm.tables[s]) for s in live)
    for min_tokens in (16, 128, 0):
        buf, _ = c.paged_decode_plan(live, H * G, mb, min_tokens)
        check_plan(bm, parse_plan(buf), live, G, min_tokens or 128)


def walk_first_piece(plan, grid, c):
    """The first piece of CTA c as the split pass walks it: units
    [c * chunk, min((c + 1) * chunk, W)), chunk = ceil(W / grid); segments
    are scanned from the first one, skipping those that end at or before the
    CTA's first unit (a linear scan, independent of the builder's search)."""
    W, B = plan["W"], plan["B"]
    chunk = max(1, -(-W // grid))
    r0 = c * chunk
    if r0 >= W:
        return None
    r1 = min(r0 + chunk, W)
    for si, s in enumerate(plan["segs"]):
        n, w = int(s["b1"] - s["b0"]), max(1, int(s["w"]))
        end_seg = int(s["wpre"]) + n * w
        if n <= 0 or r0 >= end_seg:
            continue
        end = min(r1, end_seg)
        jb, je = -(-(r0 - int(s["wpre"])) // w), -(-(end - int(s["wpre"])) // w)
        b0, b1 = int(s["b0"]) + jb, int(s["b0"]) + je
        return dict(seg=si, rep=int(s["rep"]), head=int(s["head"]), b0=b0, b1=b1,
                    tok_end=min(b1 * B, int(s["tok_end"])), ncols=int(s["ncols"]),
                    mem=int(s["mem"]), r_after=end)
    return None


@pytest.mark.parametrize("grid", [1, 7, 152, 304, 1024])
@pytest.mark.parametrize("name", ["qwen_2k", "shared_8k", "gqa70b_32k"])
def test_start_records_follow_the_walk(name, grid):
    # one record per CTA of the grid the option names: the first piece the
    # split pass's walk yields for that CTA, the position after it, and the
    # piece's first physical blocks from the member's own table
    from paged_kv_cache_65_gb300 import _lib

    wl = synth.workload(name)
    bm, c = build_both(wl)
    c.kv_pool_set_option(_lib.KV_OPT_PLAN_GRID, grid)
    mb = max(len(bm.tables[s]) for s in wl.decode_seqs)
    plan = parse_plan(c.paged_decode_plan(wl.decode_seqs, wl.n_q_heads, mb)[0])
    assert plan["start_grid"] == grid and len(plan["starts"]) == grid
    for cta in range(grid):
        R = plan["starts"][cta]
        want = walk_first_piece(plan, grid, cta)
        if want is None:
            assert R["seg"] == -1
            continue
        for k, v in want.items():
            assert int(R[k]) == v, (cta, k)
        table = bm.tables[wl.decode_seqs[want["rep"]]]
        n = min(16, want["b1"] - want["b0"], len(table) - want["b0"])
        assert int(R["n_pid"]) == n
        assert list(R["pid"][:n]) == table[want["b0"]:want["b0"] + n]


def test_plans_without_a_known_grid_have_no_start_records():
    # a pool whose device is unknown (host only) and no grid option: no records
    wl = synth.workload("qwen_2k")
    bm, c = build_both(wl)
    mb = max(len(bm.tables[s]) for s in wl.decode_seqs)
    plan = parse_plan(c.paged_decode_plan(wl.decode_seqs, wl.n_q_heads, mb)[0])
    assert plan["start_grid"] == 0 and len(plan["starts"]) == 0
    from paged_kv_cache_65_gb300 import _lib

    with pytest.raises(Exception):
        c.kv_pool_set_option(_lib.KV_OPT_PLAN_GRID, 1025)


def nested_tree(levels, B=16, fan=2, run_tokens=320, leaf_tokens=37):
    """A prompt forked into branches that each grow a long run and fork again,
    `levels` deep; returns (workload ops, leaves)."""
    ops, nxt = [("append", 0, run_tokens, 0)], 1
    frontier = [0]
    for lev in range(levels):
        new = []
        for par in frontier:
            for _ in range(fan):
                ops.append(("fork", par, nxt))
                ops.append(("append", nxt, run_tokens + 16 * lev, nxt))
                new.append(nxt)
                nxt += 1
            ops.append(("release", par))
        frontier = new
    for k, leaf in enumerate(frontier):
        ops.append(("append", leaf, leaf_tokens + k, 1000 + leaf))
    return ops, frontier


@pytest.mark.parametrize("levels,G", [(2, 4), (2, 8), (3, 2), (5, 4)])
def test_nested_forks_read_every_shared_block_once(levels, G):
    # a prompt shared by all leaves, runs shared by the leaves under each
    # branch, deeper runs under each sub-branch: every block the leaves'
    # tables name is read once per K/V head, as long as no sequence sits in
    # more than the plan's maximum of shared runs (here 3); deeper levels are
    # read by each sharer, but still exactly once per sequence
    B, H = 16, 2
    ops, leaves = nested_tree(levels, B)
    wl = synth.Workload("nested", 1, 8192, B, H * G, H, 128, "bf16", 5, None, ops, leaves)
    bm, c = build_both(wl)
    mb = max(len(bm.tables[s]) for s in leaves)
    plan = parse_plan(c.paged_decode_plan(leaves, H * G, mb)[0])
    check_plan(bm, plan, leaves, G, 128)
    distinct = {p for s in leaves for p in bm.tables[s][: -(-bm.lengths[s] // B)]}
    read = [0] * H
    for s in plan["segs"]:
        read[int(s["head"])] += int(s["b1"] - s["b0"])
    if levels <= 3:  # a leaf sits in `levels` shared runs
        assert read == [len(distinct)] * H
        # one shared segment per branch point and head (the root's prompt, then each branch)
        n_nodes = sum(2 ** k for k in range(levels))
        assert plan["n_shared_segs"] == n_nodes * H
    else:
        assert all(r > len(distinct) for r in read)  # the deepest runs are read per sharer


@pytest.mark.parametrize("dtype,B,head_dim,expect", [
    ("fp8_e4m3", 16, 128, 3), ("fp8_e4m3", 24, 128, 2), ("fp8_e4m3", 192, 128, 3),
    ("bf16", 16, 64, 2), ("q8_0", 16, 128, 2), ("bf16", 32, 128, 3)])
def test_forced_tcgen05_plans_only_where_the_pass_exists(dtype, B, head_dim, expect):
    # KV_OPT_DECODE_PATH 3 asks for tcgen05; the plan takes it for bfloat16
    # and FP8 pools with D_h = 128 and a block size whose rows fill whole
    # TMA boxes, else the warp-level pass (q8_0 pools always)
    from paged_kv_cache_65_gb300 import _lib

    H, G = 2, 4
    ops = [("append", 0, 5 * B + 3, 0), ("fork", 0, 1), ("append", 2, 3 * B, 2)]
    wl = synth.Workload("forced", 1, 64, B, H * G, H, head_dim, dtype, 5,
                        synth.permutation((5, 1), 64), ops, [0, 1, 2])
    bm, c = build_both(wl)
    c.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, 3)
    mb = max(len(bm.tables[s]) for s in wl.decode_seqs)
    buf, _ = c.paged_decode_plan(wl.decode_seqs, wl.n_q_heads, mb)
    plan = parse_plan(buf)
    assert plan["kernel"] == expect
    check_plan(bm, plan, wl.decode_seqs, G, 128)
