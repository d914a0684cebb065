"""GPU parity: the CUDA path (through the C ABI) against the oracle on the
same seeded inputs.

Integer work (slots, copy pairs, tables, pool bytes after slot writes and
copy-on-write) must be bit-exact; attention outputs must be within 1e-5
max-abs for float32 K/V and 2e-3 for bfloat16 K/V (float32 accumulation).
"""

import numpy as np
import pytest

import synth
from oracle.attention import decode_attention
from oracle.kv_store import to_f64
from oracle.runner import OracleRun

torch = pytest.importorskip("torch")
pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]

TOL = {"f32": 1e-5, "bf16": 2e-3}

# KV_OPT_DECODE_PATH: 0 automatic, 1 CUDA cores, 2 warp-level MMA, 3 tcgen05
TENSOR_PATHS = [2, 3]


def make(wl, zero=True, path=0, fill_nan=False):
    from paged_kv_cache_65_gb300 import PagedKVCache
    from paged_kv_cache_65_gb300 import _lib
    from paged_kv_cache_65_gb300.driver import DeviceRun

    cache = PagedKVCache(wl.n_layers, wl.n_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim,
                         wl.dtype, free_order=wl.free_order)
    cache.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, path)
    if fill_nan:
        cache.k.fill_(float("nan"))
        cache.v.fill_(float("nan"))
    elif zero:
        cache.k.zero_()
        cache.v.zero_()
    run = DeviceRun(cache, wl.n_q_heads)
    for op in wl.build_ops:
        run.apply(op, wl.append_values)
    return cache, run


def host_bits(t):
    from paged_kv_cache_65_gb300.driver import to_host_bits

    return to_host_bits(t)


def check_status(cache):
    assert cache.kv_pool_device_status() == 0


def max_err(gpu, ref):
    return float(np.max(np.abs(gpu.astype(np.float64) - ref))) if ref.size else 0.0


@pytest.mark.parametrize("steps", [2])
def test_tiny_full_parity(steps):
    wl = synth.workload("tiny")
    orc = OracleRun(wl)
    cache, run = make(wl)
    assert np.array_equal(host_bits(cache.k), orc.st.K)
    assert np.array_equal(host_bits(cache.v), orc.st.V)
    for step in range(steps):
        so, co, q, outs = orc.step(step)
        _, k, v = wl.step_values(step)
        sg, pg, og = run.step(wl.decode_seqs, q, k, v)
        assert list(sg) == so and [tuple(p) for p in pg] == co
        assert np.array_equal(host_bits(cache.k), orc.st.K)
        assert np.array_equal(host_bits(cache.v), orc.st.V)
        err = max_err(og.cpu().numpy()[0], outs[0])
        assert err <= TOL["f32"], err
    check_status(cache)


def test_qwen_2k_full_parity():
    wl = synth.workload("qwen_2k")
    orc = OracleRun(wl)
    cache, run = make(wl)
    for step in range(2):
        so, co, q, outs = orc.step(step)
        _, k, v = wl.step_values(step)
        sg, pg, og = run.step(wl.decode_seqs, q, k, v)
        assert list(sg) == so and len(pg) == 0
        err = max_err(og.cpu().numpy()[0], outs[0])
        assert err <= TOL["bf16"], err
    assert np.array_equal(host_bits(cache.k), orc.st.K)
    assert np.array_equal(host_bits(cache.v), orc.st.V)
    check_status(cache)


def attend_four_ways(cache, run, wl, qh):
    """The same step's attention per sequence and through the sharing-aware
    plan, each on the warp-level MMA pass (2) and on tcgen05 (3); the
    bench's launch configuration is the planned pass."""
    from paged_kv_cache_65_gb300 import _lib

    d_table, d_lens, mb = run.tables(wl.decode_seqs)
    qd = torch.from_numpy(qh.view(np.int16)).cuda().view(torch.bfloat16)
    outs = {}
    for path in TENSOR_PATHS:
        cache.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, path)
        outs[("plain", path)] = run.attend(0, qd, d_table, mb, d_lens,
                                           len(wl.decode_seqs)).cpu().numpy()
        h_plan, d_plan, ws_bytes = run.plan(wl.decode_seqs, mb)
        outs[("planned", path)] = run.attend_planned(0, qd, d_table, mb, h_plan, d_plan,
                                                     ws_bytes).cpu().numpy()
    return outs


def test_shared_8k_full_parity():
    # all 16 sequences, every output, four ways
    wl = synth.workload("shared_8k")
    orc = OracleRun(wl)
    cache, run = make(wl)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    sg, pg = run.reserve(wl.decode_seqs)
    assert list(sg) == so and len(pg) == 0
    run.write(sg, pg, k, v)
    ref = orc.attend(0, qh)
    for key, got in attend_four_ways(cache, run, wl, qh).items():
        assert max_err(got, ref) <= TOL["bf16"], key
    # the 384 shared prefix blocks are read by all 16 sequences: bit-identical pools
    assert np.array_equal(host_bits(cache.k), orc.st.K)
    assert np.array_equal(host_bits(cache.v), orc.st.V)
    check_status(cache)


def test_gqa70b_32k_cow_and_full_parity():
    # all 48 branches on both steps (the first copies 48 shared tails), four ways
    wl = synth.workload("gqa70b_32k")
    orc = OracleRun(wl)
    cache, run = make(wl)
    for step in range(2):
        so, co = orc.reserve_step()
        qh = orc.write_step(step, so, co)
        _, k, v = wl.step_values(step)
        sg, pg = run.reserve(wl.decode_seqs)
        assert list(sg) == so
        assert [tuple(p) for p in pg] == co
        assert len(co) == (48 if step == 0 else 0)
        run.write(sg, pg, k, v)
        if step == 0:
            kd = host_bits(cache.k)
            for src, dst in co:
                assert np.array_equal(kd[:, dst], orc.st.K[:, dst])
                # the copy kept the shared tokens and the new token went to the copy
                assert np.array_equal(kd[:, dst, :3], kd[:, src, :3])
            assert np.array_equal(kd, orc.st.K)
            assert np.array_equal(host_bits(cache.v), orc.st.V)
        ref = orc.attend(0, qh)
        for key, got in attend_four_ways(cache, run, wl, qh).items():
            assert max_err(got, ref) <= TOL["bf16"], (step, key)
    check_status(cache)


def ragged_workload(dtype, D, G, B, lens, H_kv=2, seed=0, n_blocks=None):
    """Independent sequences of the given lengths after one decode step."""
    n_blocks = n_blocks or sum(-(-l // B) for l in lens) + len(lens) + 3
    ops = [("append", s, l - 1, s) for s, l in enumerate(lens) if l > 1]
    return synth.Workload("ragged", 1, n_blocks, B, H_kv * G, H_kv, D, dtype, seed,
                          synth.permutation((seed, 9), n_blocks), ops, list(range(len(lens))))


SHAPES = [
    ("f32", 64, 4, 4), ("f32", 64, 1, 2), ("f32", 128, 8, 16), ("f32", 128, 2, 1),
    ("bf16", 128, 4, 16), ("bf16", 128, 8, 16), ("bf16", 128, 1, 8), ("bf16", 128, 2, 32),
    ("bf16", 64, 4, 16), ("bf16", 64, 8, 64), ("bf16", 128, 4, 3), ("bf16", 128, 4, 64),
    ("f32", 64, 8, 5),
]


CASES = ([s + (0,) for s in SHAPES]
         + [s + (p,) for p in (1, 2) for s in SHAPES if s[0] == "bf16" and s[3] % 8 == 0]
         + [s + (3,) for s in SHAPES if s[0] == "bf16" and s[3] % 8 == 0 and s[1] == 128])


@pytest.mark.parametrize("dtype,D,G,B,path", CASES)
def test_ragged_shapes(dtype, D, G, B, path):
    # path 0: automatic; 1: CUDA cores; 2: warp-level MMA; 3: tcgen05
    lens = [1, 2, B - 1 if B > 1 else 3, B, B + 1, 3 * B + 2, 97, 700]
    lens = [max(1, l) for l in lens]
    wl = ragged_workload(dtype, D, G, B, lens, seed=D + G + B)
    orc = OracleRun(wl)
    cache, run = make(wl, path=path)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    sg, pg, og = run.step(wl.decode_seqs, qh, k, v)
    assert list(sg) == so
    ref = orc.attend(0, qh)
    assert max_err(og.cpu().numpy()[0], ref) <= TOL[dtype]
    check_status(cache)


def test_block_size_two_lengths_one_to_five():
    # "PagedAttention 的块表与碎片控制" §13: block size 2 with lengths 1..5
    wl = ragged_workload("f32", 64, 4, 2, [1, 2, 3, 4, 5], seed=5)
    orc = OracleRun(wl)
    cache, run = make(wl)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    _, _, og = run.step(wl.decode_seqs, qh, k, v)
    assert max_err(og.cpu().numpy()[0], orc.attend(0, qh)) <= 1e-5
    assert np.array_equal(host_bits(cache.k), orc.st.K)


def test_single_token_context_returns_value_exactly():
    wl = ragged_workload("f32", 64, 4, 4, [1, 1, 1])
    cache, run = make(wl)
    q, k, v = wl.step_values(0)
    _, _, og = run.step(wl.decode_seqs, q, k, v)
    got = og.cpu().numpy()[0]
    for s in range(3):
        for h in range(8):
            assert np.array_equal(got[s, h], v[0, s, h // 4])


def test_empty_context_gives_zeros_and_others_unchanged():
    wl = ragged_workload("bf16", 128, 4, 16, [40, 17, 300])
    orc = OracleRun(wl)
    cache, run = make(wl)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    run.write(*run.reserve(wl.decode_seqs), k, v)
    d_table, d_lens, mb = run.tables(wl.decode_seqs)
    d_lens[1] = 0
    qd = torch.from_numpy(qh.view(np.int16)).cuda().view(torch.bfloat16)
    out = run.attend(0, qd, d_table, mb, d_lens, 3)
    got = out.cpu().numpy()
    ref = orc.attend(0, qh)
    assert not got[1].any()
    assert max_err(got[[0, 2]], ref[[0, 2]]) <= TOL["bf16"]


def test_placement_invariance_and_determinism():
    outs = []
    for order_seed in (1, 2):
        wl = ragged_workload("bf16", 128, 4, 16, [33, 1000, 2049, 5], seed=3)
        wl.free_order = synth.permutation((order_seed, 77), wl.n_blocks)
        cache, run = make(wl)
        q, k, v = wl.step_values(0)
        _, _, og = run.step(wl.decode_seqs, q, k, v)
        d_table, d_lens, mb = run.tables(wl.decode_seqs)
        qd = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
        again = run.attend(0, qd, d_table, mb, d_lens, 4)
        assert torch.equal(again, og[0])
        outs.append(og.cpu())
    assert torch.equal(outs[0], outs[1])


def test_split_and_merge_calls_equal_one_call():
    wl = ragged_workload("bf16", 128, 8, 16, [5000, 3, 800], seed=4)
    cache, run = make(wl)
    q, k, v = wl.step_values(0)
    _, _, og = run.step(wl.decode_seqs, q, k, v)
    d_table, d_lens, mb = run.tables(wl.decode_seqs)
    qd = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    ws = run.workspace(3)
    out = torch.empty_like(og[0])
    cache.paged_decode_partials(0, qd, wl.n_q_heads, d_table, mb, d_lens, 3, ws)
    cache.paged_decode_merge(wl.n_q_heads, d_lens, 3, out, ws)
    assert torch.equal(out, og[0])


def test_bf16_output():
    wl = ragged_workload("bf16", 128, 4, 16, [100, 2000], seed=6)
    orc = OracleRun(wl)
    cache, run = make(wl)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    run.write(*run.reserve(wl.decode_seqs), k, v)
    d_table, d_lens, mb = run.tables(wl.decode_seqs)
    qd = torch.from_numpy(qh.view(np.int16)).cuda().view(torch.bfloat16)
    out = run.attend(0, qd, d_table, mb, d_lens, 2, out_dtype=torch.bfloat16)
    got = out.float().cpu().numpy()
    ref = orc.attend(0, qh)
    assert np.all(np.abs(got - ref) <= 2e-3 + np.abs(ref) * 2.0 ** -8)


def host_buffer(a, pinned):
    """A caller's host buffer: the NumPy array itself (pageable: the step copies
    it through its staging area), or a page-locked copy that the device
    addresses in place (new K / V read and outputs written through the
    mapping)."""
    if not pinned:
        return a
    flat = a.view(np.int16) if a.dtype == np.uint16 else a
    return torch.from_numpy(np.ascontiguousarray(flat)).pin_memory()


def host_out(shape, pinned):
    if not pinned:
        return np.zeros(shape, dtype=np.float32)
    return torch.zeros(shape, dtype=torch.float32).pin_memory()


def as_np(out):
    return out if isinstance(out, np.ndarray) else out.numpy()


@pytest.mark.parametrize("pinned", [False, True])
def test_multilayer_decode_step_host_buffers(pinned):
    # the whole-step C entry point with host buffers, 3 layers, shared prefix
    L, B, H, G, D = 3, 8, 2, 4, 128
    # sequences 0 and 1 share a prefix whose tail block holds 3 of 8 slots:
    # step 0 makes 0 copy it and lets 1 write in place
    ops = [("append", 100, 43, 0), ("fork", 100, 0), ("fork", 100, 1), ("release", 100),
           ("append", 2, 77, 2)]
    wl = synth.Workload("multi", L, 64, B, H * G, H, D, "bf16", 8,
                        synth.permutation((8, 1), 64), ops, [0, 1, 2])
    orc = OracleRun(wl)
    from paged_kv_cache_65_gb300 import PagedKVCache
    from paged_kv_cache_65_gb300.driver import DeviceRun

    cache = PagedKVCache(L, 64, B, H, D, "bf16", free_order=wl.free_order)
    cache.k.zero_()
    cache.v.zero_()
    run = DeviceRun(cache, H * G)
    for op in wl.build_ops:
        run.apply(op, wl.append_values)
    max_blocks = 16
    staging = torch.empty(cache.kv_decode_step_staging_bytes(3, H * G, max_blocks),
                          dtype=torch.uint8, device="cuda")
    for step in range(3):
        so, co = orc.reserve_step()
        assert len(co) == (1 if step == 0 else 0)
        q = orc.write_step(step, so, co)
        qL = np.ascontiguousarray(np.broadcast_to(q, (L,) + q.shape))
        _, k, v = wl.step_values(step)
        out = host_out((L, 3, H * G, D), pinned)
        cache.kv_decode_step_host([0, 1, 2], H * G, max_blocks, host_buffer(qL, pinned),
                                  host_buffer(k, pinned), host_buffer(v, pinned), out, staging)
        for layer in range(L):
            ref = orc.attend(layer, q)
            assert max_err(as_np(out)[layer], ref) <= TOL["bf16"]
    assert np.array_equal(host_bits(cache.k), orc.st.K)
    assert np.array_equal(host_bits(cache.v), orc.st.V)
    check_status(cache)


def test_device_checks_flag_bad_ids_without_faulting():
    wl = ragged_workload("bf16", 128, 4, 16, [40, 50])
    cache, run = make(wl)
    q, k, v = wl.step_values(0)
    run.step(wl.decode_seqs, q, k, v)
    d_table, d_lens, mb = run.tables(wl.decode_seqs)
    d_table[0, 0] = wl.n_blocks + 5  # out of range: the kernel substitutes block 0
    qd = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    run.attend(0, qd, d_table, mb, d_lens, 2)
    assert cache.kv_pool_device_status() & 1
    bad = torch.tensor([wl.n_blocks * 16 + 3], dtype=torch.int64, device="cuda")
    kk = torch.zeros((1, 1, 2, 128), dtype=torch.bfloat16, device="cuda")
    cache.reshape_and_cache(0, kk, kk, bad, 1)
    assert cache.kv_pool_device_status() & 2
    assert cache.kv_pool_device_status() == 0


@pytest.mark.parametrize("path", [0, 1, 2, 3])
def test_unused_slots_holding_nan_do_not_leak(path):
    # the pool starts as NaN bit patterns: slots past each context in the last
    # block are loaded with the block but must not reach any output
    wl = ragged_workload("bf16", 128, 4, 16, [1, 5, 17, 33, 250, 1000], seed=12)
    orc = OracleRun(wl)
    cache, run = make(wl, fill_nan=True, path=path)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    _, _, og = run.step(wl.decode_seqs, qh, k, v)
    got = og.cpu().numpy()[0]
    assert np.isfinite(got).all()
    assert max_err(got, orc.attend(0, qh)) <= TOL["bf16"]


@pytest.mark.parametrize("name", ["qwen_2k", "gqa70b_32k"])
def test_tensor_core_and_cuda_core_paths_agree(name):
    wl = synth.workload(name)
    if name == "gqa70b_32k":
        wl.build_ops = wl.build_ops[:10]  # two parents, eight branches: keeps the test short
        wl.decode_seqs = wl.decode_seqs[:8]
    outs = []
    for path in (1, 2, 3):
        cache, run = make(wl, zero=False, path=path)
        q, k, v = wl.step_values(0)
        _, _, og = run.step(wl.decode_seqs, q, k, v)
        outs.append(og.cpu().numpy())
        del cache, run
        torch.cuda.empty_cache()
    for o in outs[1:]:
        assert float(np.max(np.abs(outs[0] - o))) <= 2e-3


# ---------------------------------------------------------------- planned
# The sharing-aware pass: shared prefix blocks are read once for all sharers.


@pytest.mark.parametrize("path", TENSOR_PATHS)
@pytest.mark.parametrize("seed,G,B", [(0, 1, 16), (1, 2, 8), (2, 4, 16), (3, 8, 16), (4, 4, 8),
                                      (5, 8, 32), (6, 4, 64)])
def test_planned_random_fork_trees_against_oracle(seed, G, B, path):
    rng = np.random.default_rng(seed)
    H = 2
    ops, live, nxt = [], [], 0
    for _ in range(4):
        ops.append(("append", nxt, int(rng.integers(100, 700)), nxt))
        live.append(nxt)
        nxt += 1
    for _ in range(14):
        p = int(rng.choice(live))
        if rng.random() < 0.6:
            ops.append(("fork", p, nxt))
            live.append(nxt)
            nxt += 1
        else:
            ops.append(("append", p, int(rng.integers(1, 200)), 1000 + nxt + len(ops)))
    wl = synth.Workload("forks", 1, 2048, B, H * G, H, 128, "bf16", seed,
                        synth.permutation((seed, 5), 2048), ops, live)
    orc = OracleRun(wl)
    cache, run = make(wl, path=path)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    sg, pg, og = run.step(wl.decode_seqs, qh, k, v, planned=True)
    assert list(sg) == so and [tuple(p) for p in pg] == co
    h_plan, _, _ = run.plan(wl.decode_seqs, run.max_blocks(wl.decode_seqs))
    from paged_kv_cache_65_gb300.cache import parse_plan

    assert parse_plan(h_plan)["n_shared_segs"] > 0  # the trees do share prefixes
    assert max_err(og.cpu().numpy()[0], orc.attend(0, qh)) <= TOL["bf16"]
    check_status(cache)


@pytest.mark.parametrize("path", TENSOR_PATHS)
@pytest.mark.parametrize("levels,G", [(2, 4), (3, 8), (4, 2)])
def test_planned_nested_forks_against_oracle(levels, G, path):
    # a prompt forked into branches that grow and fork again: the plan reads
    # the prompt once for all leaves, each branch's run once for its leaves
    # (up to three shared runs per sequence; deeper ones privately)
    from test_plan import nested_tree

    B, H = 16, 2
    ops, leaves = nested_tree(levels, B, run_tokens=200, leaf_tokens=21)
    wl = synth.Workload("nested", 1, 2048, B, H * G, H, 128, "bf16", 40 + levels,
                        synth.permutation((40 + levels, 5), 2048), ops, leaves)
    orc = OracleRun(wl)
    cache, run = make(wl, path=path)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    sg, pg, og = run.step(wl.decode_seqs, qh, k, v, planned=True)
    assert list(sg) == so and [tuple(p) for p in pg] == co
    h_plan, _, _ = run.plan(wl.decode_seqs, run.max_blocks(wl.decode_seqs))
    from paged_kv_cache_65_gb300.cache import parse_plan

    assert parse_plan(h_plan)["n_shared_segs"] >= (2 ** min(levels, 3) - 1) * H
    assert max_err(og.cpu().numpy()[0], orc.attend(0, qh)) <= TOL["bf16"]
    check_status(cache)


@pytest.mark.parametrize("path", TENSOR_PATHS)
def test_planned_equals_plain_without_sharing(path):
    wl = synth.workload("qwen_2k")
    cache, run = make(wl, zero=False, path=path)
    q, k, v = wl.step_values(0)
    run.write(*run.reserve(wl.decode_seqs), k, v)
    d_table, d_lens, mb = run.tables(wl.decode_seqs)
    qd = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    h_plan, d_plan, ws_bytes = run.plan(wl.decode_seqs, mb)
    a = run.attend_planned(0, qd, d_table, mb, h_plan, d_plan, ws_bytes).clone()
    b = run.attend(0, qd, d_table, mb, d_lens, len(wl.decode_seqs))
    assert float((a - b).abs().max()) <= 1e-6


@pytest.mark.parametrize("path", TENSOR_PATHS)
@pytest.mark.parametrize("name", ["shared_8k", "gqa70b_32k"])
def test_planned_start_records_change_no_bit(name, path):
    # the same step twice on identical pools: once with the plan's per-CTA
    # start records built for the launch's grid (the kernels take their first
    # pieces and block ids from them), once with records built for another
    # grid (ignored: the kernels search the plan); the outputs are identical
    from paged_kv_cache_65_gb300 import _lib
    from paged_kv_cache_65_gb300.cache import parse_plan

    wl = synth.workload(name)
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    outs = []
    for grid in (0, 7):
        cache, run = make(wl, zero=False, path=path)
        cache.kv_pool_set_option(_lib.KV_OPT_PLAN_GRID, grid)
        q, k, v = wl.step_values(0)
        _, _, og = run.step(wl.decode_seqs, q, k, v, planned=True)
        plan = parse_plan(run.plan(wl.decode_seqs, run.max_blocks(wl.decode_seqs))[0])
        if grid == 0:
            assert plan["start_grid"] == (sm if plan["kernel"] == 3 else 2 * sm)
        else:
            assert plan["start_grid"] == 7
        outs.append(og.cpu().numpy())
        check_status(cache)
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("pinned", [False, True])
@pytest.mark.parametrize("path", TENSOR_PATHS)
def test_multilayer_host_step_with_long_shared_prefix(path, pinned):
    # kv_decode_step_host plans the step: sequences 0-2 share 300 tokens
    L, B, H, G, D = 2, 16, 2, 4, 128
    ops = [("append", 100, 300, 0), ("fork", 100, 0), ("fork", 100, 1), ("fork", 100, 2),
           ("release", 100), ("append", 1, 20, 1), ("append", 3, 77, 2)]
    wl = synth.Workload("multi_shared", L, 128, B, H * G, H, D, "bf16", 9,
                        synth.permutation((9, 1), 128), ops, [0, 1, 2, 3])
    orc = OracleRun(wl)
    from paged_kv_cache_65_gb300 import PagedKVCache
    from paged_kv_cache_65_gb300.driver import DeviceRun

    from paged_kv_cache_65_gb300 import _lib

    cache = PagedKVCache(L, 128, B, H, D, "bf16", free_order=wl.free_order)
    cache.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, path)
    cache.k.zero_()
    cache.v.zero_()
    run = DeviceRun(cache, H * G)
    for op in wl.build_ops:
        run.apply(op, wl.append_values)
    max_blocks = 32
    staging = torch.empty(cache.kv_decode_step_staging_bytes(4, H * G, max_blocks),
                          dtype=torch.uint8, device="cuda")
    for step in range(2):
        so, co = orc.reserve_step()
        q = orc.write_step(step, so, co)
        qL = np.ascontiguousarray(np.broadcast_to(q, (L,) + q.shape))
        _, k, v = wl.step_values(step)
        out = host_out((L, 4, H * G, D), pinned)
        cache.kv_decode_step_host([0, 1, 2, 3], H * G, max_blocks, host_buffer(qL, pinned),
                                  host_buffer(k, pinned), host_buffer(v, pinned), out, staging)
        for layer in range(L):
            assert max_err(as_np(out)[layer], orc.attend(layer, q)) <= TOL["bf16"]
    check_status(cache)


@pytest.mark.parametrize("path", TENSOR_PATHS)
def test_single_layer_host_step_page_locked_and_pageable_agree(path):
    # one layer (the outputs come back in one piece): the same three steps,
    # two copy-on-write copies among them, through page-locked buffers (new K / V
    # read in place, outputs written in place) and through pageable ones
    # (staging copies) give the same bits in the outputs and the pools, and
    # match the oracle
    B, H, G, D = 16, 2, 4, 128
    ops = [("append", 100, 150, 0), ("fork", 100, 0), ("fork", 100, 1), ("append", 2, 700, 1),
           ("append", 3, 31, 2)]
    wl = synth.Workload("host_step", 1, 160, B, H * G, H, D, "bf16", 12,
                        synth.permutation((12, 1), 160), ops, [0, 1, 2, 3, 100])
    from paged_kv_cache_65_gb300 import PagedKVCache, _lib
    from paged_kv_cache_65_gb300.driver import DeviceRun

    results = []
    for pinned in (False, True):
        orc = OracleRun(wl)
        cache = PagedKVCache(1, 160, B, H, D, "bf16", free_order=wl.free_order)
        cache.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, path)
        cache.k.zero_()
        cache.v.zero_()
        run = DeviceRun(cache, H * G)
        for op in wl.build_ops:
            run.apply(op, wl.append_values)
        n, max_blocks = len(wl.decode_seqs), 64
        staging = torch.empty(cache.kv_decode_step_staging_bytes(n, H * G, max_blocks),
                              dtype=torch.uint8, device="cuda")
        outs = []
        for step in range(3):
            so, co = orc.reserve_step()
            assert len(co) == (2 if step == 0 else 0)  # the shared tail, for 0 and 1
            q = orc.write_step(step, so, co)
            _, k, v = wl.step_values(step)
            out = host_out((1, n, H * G, D), pinned)
            cache.kv_decode_step_host(wl.decode_seqs, H * G, max_blocks,
                                      host_buffer(q[None], pinned), host_buffer(k, pinned),
                                      host_buffer(v, pinned), out, staging)
            got = as_np(out).copy()
            assert max_err(got[0], orc.attend(0, q)) <= TOL["bf16"]
            outs.append(got)
        assert np.array_equal(host_bits(cache.k), orc.st.K)
        assert np.array_equal(host_bits(cache.v), orc.st.V)
        check_status(cache)
        results.append(outs)
    for a, b in zip(*results):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("path", TENSOR_PATHS)
@pytest.mark.parametrize("planned", [False, True])
def test_programmatic_launch_gives_identical_results(planned, path):
    # the same step with and without programmatic dependent launches
    from paged_kv_cache_65_gb300 import _lib

    outs = []
    for pdl in (1, 0):
        wl = ragged_workload("bf16", 128, 4, 16, [33, 1000, 2049, 5, 700], seed=31)
        cache, run = make(wl, path=path)
        cache.kv_pool_set_option(_lib.KV_OPT_PDL, pdl)
        q, k, v = wl.step_values(0)
        _, _, og = run.step(wl.decode_seqs, q, k, v, planned=planned)
        outs.append(og.cpu())
    assert torch.equal(outs[0], outs[1])


class RampWorkload(synth.Workload):
    """Keys whose scale grows along each appended run (0.25 at its start, 4
    at its end): the largest score of a query keeps rising deep into the
    context, so the running maximum moves in late stages of a piece, not only
    in its first one."""

    def append_values(self, value_seed, n_tokens):
        k, v = super().append_values(value_seed, n_tokens)
        ramp = np.linspace(0.25, 4.0, n_tokens, dtype=np.float32)[None, :, None, None]
        if self.dtype == "bf16":
            kf = (k.astype(np.uint32) << 16).view(np.float32)
            k = synth.storage_values(np.ascontiguousarray(kf * ramp), "bf16")
        else:
            k = np.ascontiguousarray(k * ramp)
        return k, v


@pytest.mark.parametrize("path", TENSOR_PATHS + [1])
@pytest.mark.parametrize("planned", [False, True])
def test_rising_scores_move_the_maximum_inside_pieces(path, planned):
    G, H, B = 4, 2, 16
    ops = [("append", 0, 3000, 0), ("fork", 0, 1), ("fork", 0, 2), ("append", 1, 500, 1),
           ("append", 3, 1800, 2), ("append", 4, 4100, 3)]
    wl = RampWorkload("ramp", 1, 1024, B, H * G, H, 128, "bf16", 21,
                      synth.permutation((21, 2), 1024), ops, [0, 1, 2, 3, 4])
    orc = OracleRun(wl)
    cache, run = make(wl, path=path)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    _, _, og = run.step(wl.decode_seqs, qh, k, v, planned=planned and path != 1)
    assert max_err(og.cpu().numpy()[0], orc.attend(0, qh)) <= TOL["bf16"]
    check_status(cache)


# ----------------------------------------------------------- maximum sizes


@pytest.mark.parametrize("path", TENSOR_PATHS)
def test_one_sequence_of_128k_tokens(path):
    # a single 131,072-token context (8,192 blocks of 16) at G = 8: the whole
    # grid's work is one segment per K/V head, cut into many pieces that the
    # merge recombines; plain and planned, against the oracle
    n = 131072
    wl = ragged_workload("bf16", 128, 8, 16, [n], H_kv=8, seed=77, n_blocks=n // 16 + 8)
    orc = OracleRun(wl)
    cache, run = make(wl, zero=False, path=path)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    run.write(*run.reserve(wl.decode_seqs), k, v)
    ref = orc.attend(0, qh)
    d_table, d_lens, mb = run.tables(wl.decode_seqs)
    qd = torch.from_numpy(qh.view(np.int16)).cuda().view(torch.bfloat16)
    got = run.attend(0, qd, d_table, mb, d_lens, 1).cpu().numpy()
    assert max_err(got, ref) <= TOL["bf16"]
    h_plan, d_plan, ws_bytes = run.plan(wl.decode_seqs, mb)
    got = run.attend_planned(0, qd, d_table, mb, h_plan, d_plan, ws_bytes).cpu().numpy()
    assert max_err(got, ref) <= TOL["bf16"]
    check_status(cache)


@pytest.mark.parametrize("path", TENSOR_PATHS)
def test_a_thousand_short_sequences(path):
    # 1,024 sequences in one batch (more segments than CTAs by far): lengths
    # 1 to 300, a third of them forked from one 200-token prompt; every
    # output against the oracle, plain and planned
    rng = np.random.default_rng(5)
    ops, seqs = [("append", 5000, 200, 0)], []
    for s in range(1024):
        if s % 3 == 0:
            ops.append(("fork", 5000, s))
            extra = int(rng.integers(0, 60))
        else:
            extra = int(rng.integers(0, 300))
        if extra:
            ops.append(("append", s, extra, 1 + s))
        seqs.append(s)
    wl = synth.Workload("thousand", 1, 12288, 16, 32, 8, 128, "bf16", 88,
                        synth.permutation((88, 1), 12288), ops, seqs)
    orc = OracleRun(wl)
    cache, run = make(wl, path=path)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    sg, pg = run.reserve(seqs)
    assert list(sg) == so and [tuple(p) for p in pg] == co
    run.write(sg, pg, k, v)
    ref = orc.attend(0, qh)
    for key, got in attend_four_ways(cache, run, wl, qh).items():
        if key[1] == path:
            assert max_err(got, ref) <= TOL["bf16"], key
    assert np.array_equal(host_bits(cache.k), orc.st.K)
    check_status(cache)
