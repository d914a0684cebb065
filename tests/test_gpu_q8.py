"""q8_0 pools on the GPU against the oracle ("第 8 章 推理优化" §8.4.2, Fig.
8-23: 32 values share one fp16 scale, one int8 code each): the codes and
scales the slot write stores and the blocks copy-on-write copies are
bit-exact; decode attention (plain and planned, warp-level MMA pass) matches
the oracle's attention over the dequantized values within the bf16
tolerance."""

import numpy as np
import pytest

import synth
from oracle.runner import OracleRun

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TOL = 2e-3


def make(wl, code_fill=0, scale_fill=0):
    from paged_kv_cache_65_gb300 import PagedKVCache
    from paged_kv_cache_65_gb300.driver import DeviceRun

    cache = PagedKVCache(wl.n_layers, wl.n_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim,
                         wl.dtype, free_order=wl.free_order)
    cache.k.fill_(code_fill)
    cache.v.fill_(code_fill)
    cache.k_sc.view(torch.int16).fill_(scale_fill)
    cache.v_sc.view(torch.int16).fill_(scale_fill)
    run = DeviceRun(cache, wl.n_q_heads)
    for op in wl.build_ops:
        run.apply(op, wl.append_values)
    return cache, run


def same_pool(cache, st):
    """Codes and scales of the device pool equal the oracle store's, bit for
    bit (device scales are [L, N, H, B, D/32], the oracle's [L, N, B, H,
    D/32])."""
    k_sc = cache.k_sc.cpu().numpy().view(np.uint16).transpose(0, 1, 3, 2, 4)
    v_sc = cache.v_sc.cpu().numpy().view(np.uint16).transpose(0, 1, 3, 2, 4)
    return (np.array_equal(cache.k.cpu().numpy(), st.K) and np.array_equal(k_sc, st.Ks)
            and np.array_equal(cache.v.cpu().numpy(), st.V) and np.array_equal(v_sc, st.Vs))


def max_err(gpu, ref):
    return float(np.max(np.abs(gpu.astype(np.float64) - ref))) if ref.size else 0.0


def q8_workload(name, G, B, seed, ctxs, H=2, n_blocks=None, fork=None):
    n_blocks = n_blocks or (sum(-(-c // B) for c in ctxs) + 2 * len(ctxs)
                            + (-(-fork // B) + 6 if fork else 0) + 8)
    ops = [("append", s, c - 1, s) for s, c in enumerate(ctxs) if c > 1]
    seqs = list(range(len(ctxs)))
    if fork is not None:  # a prefix of `fork` tokens forked into two, parent alive
        ops += [("append", 100, fork, 99), ("fork", 100, 101), ("fork", 100, 102)]
        seqs += [100, 101, 102]
    return synth.Workload(name, 1, n_blocks, B, H * G, H, 128, "q8_0", seed,
                          synth.permutation((seed, 9), n_blocks), ops, seqs)


def test_q8_codes_scales_cow_and_outputs():
    # two steps; the first copies the shared, partly filled tail of a fork
    wl = q8_workload("q8_small", 4, 16, 21, [1, 15, 16, 17, 70, 333], fork=150)
    orc = OracleRun(wl)
    cache, run = make(wl)
    assert same_pool(cache, orc.st)  # the build's writes, quantized on the device
    for step in range(2):
        so, co, q, outs = orc.step(step)
        _, k, v = wl.step_values(step)
        sg, pg, og = run.step(wl.decode_seqs, q, k, v)
        assert list(sg) == so and [tuple(p) for p in pg] == co
        if step == 0:
            assert len(co) == 2  # 100 and 101 copy the shared tail, 102 writes in place
        assert same_pool(cache, orc.st)
        assert max_err(og.cpu().numpy()[0], outs[0]) <= TOL
    assert cache.kv_pool_device_status() == 0


def test_q8_planned_pass_with_a_shared_prefix():
    wl = q8_workload("q8_fork", 4, 16, 22, [40, 300], fork=200)
    orc = OracleRun(wl)
    cache, run = make(wl)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    sg, pg, og = run.step(wl.decode_seqs, qh, k, v, planned=True)
    assert list(sg) == so and [tuple(p) for p in pg] == co
    from paged_kv_cache_65_gb300.cache import parse_plan

    h_plan, _, _ = run.plan(wl.decode_seqs, run.max_blocks(wl.decode_seqs))
    plan = parse_plan(h_plan)
    assert plan["kernel"] == 2 and plan["n_shared_segs"] > 0
    assert max_err(og.cpu().numpy()[0], orc.attend(0, qh)) <= TOL
    assert same_pool(cache, orc.st)
    assert cache.kv_pool_device_status() == 0


@pytest.mark.parametrize("G,B", [(1, 16), (2, 8), (4, 32), (8, 64), (8, 16)])
def test_q8_ragged_shapes(G, B):
    ctxs = [1, 2, B - 1, B, B + 1, 3 * B + 2, 97, 700]
    wl = q8_workload("q8_ragged", G, B, 30 + G + B, ctxs)
    orc = OracleRun(wl)
    cache, run = make(wl)
    so, co, q, outs = orc.step(0)
    _, k, v = wl.step_values(0)
    sg, _, og = run.step(wl.decode_seqs, q, k, v)
    assert list(sg) == so
    assert same_pool(cache, orc.st)
    assert max_err(og.cpu().numpy()[0], outs[0]) <= TOL, (G, B)
    assert cache.kv_pool_device_status() == 0


def test_q8_unused_slots_with_nan_scales_do_not_leak():
    # every unused slot holds code bytes 0x7F and scales with NaN bits
    wl = q8_workload("q8_nan", 4, 16, 23, [1, 15, 17, 70, 333])
    orc = OracleRun(wl)
    cache, run = make(wl, code_fill=0x7F, scale_fill=-1)  # 0xFFFF: an fp16 NaN
    so, co, q, outs = orc.step(0)
    _, k, v = wl.step_values(0)
    _, _, og = run.step(wl.decode_seqs, q, k, v)
    got = og.cpu().numpy()[0]
    assert np.isfinite(got).all()
    assert max_err(got, outs[0]) <= TOL


def test_q8_qwen_2k_full():
    # every output of all 37 sequences, per sequence and through the plan
    from paged_kv_cache_65_gb300.driver import to_device

    wl = synth.workload("qwen_2k_q8")
    orc = OracleRun(wl)
    cache, run = make(wl)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    sg, _, og = run.step(wl.decode_seqs, qh, k, v)
    assert list(sg) == so
    ref = orc.attend(0, qh)
    assert max_err(og.cpu().numpy()[0], ref) <= TOL
    d_table, _, mb = run.tables(wl.decode_seqs)
    h_plan, d_plan, ws = run.plan(wl.decode_seqs, mb)
    got = run.attend_planned(0, to_device(qh, "bf16", "cuda"), d_table, mb, h_plan, d_plan, ws)
    assert max_err(got.cpu().numpy(), ref) <= TOL
    assert same_pool(cache, orc.st)
    assert cache.kv_pool_device_status() == 0


def test_q8_pool_without_scale_arrays_is_refused():
    from paged_kv_cache_65_gb300 import PagedKVCache, _lib
    from paged_kv_cache_65_gb300._lib import KVError

    k = torch.zeros((1, 8, 16, 2, 128), dtype=torch.uint8, device="cuda")
    v = torch.zeros_like(k)
    c2 = PagedKVCache(1, 8, 16, 2, 128, "q8_0", allocate=False, k_cache=k, v_cache=v)
    slots = torch.zeros(1, dtype=torch.int64, device="cuda")
    rows = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(KVError) as e:
        c2.reshape_and_cache(0, rows, rows, slots, 1)
    assert e.value.status == _lib.KV_ERR_INVALID_ARG
