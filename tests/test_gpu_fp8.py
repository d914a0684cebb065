"""FP8 (E4M3) pools on the GPU against the oracle: the codes the slot write
stores and the blocks copy-on-write copies are bit-exact; decode attention
(plain and planned, on the warp-level MMA pass and on the tcgen05 pass,
whose converter warps turn the codes into fp16 tiles) matches the oracle's
attention over the dequantized values within the bf16 tolerance."""

import numpy as np
import pytest

import synth
from oracle.runner import OracleRun

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TOL = 2e-3


# KV_OPT_DECODE_PATH: 0 automatic, 2 warp-level MMA, 3 tcgen05
def make(wl, fill=0, path=0):
    from paged_kv_cache_65_gb300 import PagedKVCache, _lib
    from paged_kv_cache_65_gb300.driver import DeviceRun

    cache = PagedKVCache(wl.n_layers, wl.n_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim,
                         wl.dtype, free_order=wl.free_order)
    cache.kv_pool_set_fp8_scales(wl.k_scale, wl.v_scale)
    cache.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, path)
    cache.k.fill_(fill)
    cache.v.fill_(fill)
    run = DeviceRun(cache, wl.n_q_heads)
    for op in wl.build_ops:
        run.apply(op, wl.append_values)
    return cache, run


def nan_code_equal(a, b):
    """Byte-identical, except that any two E4M3 NaN codes (0x7F, 0xFF) match."""
    na = (a & 0x7F) == 0x7F
    nb = (b & 0x7F) == 0x7F
    return bool(np.array_equal(na, nb) and np.array_equal(a[~na], b[~nb]))


def max_err(gpu, ref):
    return float(np.max(np.abs(gpu.astype(np.float64) - ref))) if ref.size else 0.0


def fp8_workload(name, G, B, seed, ctxs, k_scale=1.0, v_scale=1.0, n_blocks=256):
    H = 2
    ops = [("append", s, c - 1, s) for s, c in enumerate(ctxs) if c > 1]
    return synth.Workload(name, 1, n_blocks, B, H * G, H, 128, "fp8_e4m3", seed,
                          synth.permutation((seed, 9), n_blocks), ops, list(range(len(ctxs))),
                          k_scale=k_scale, v_scale=v_scale)


def test_fp8_small_codes_cow_and_outputs():
    wl = synth.workload("fp8_small")
    orc = OracleRun(wl)
    cache, run = make(wl)
    # the build's writes (values quantized on the device) are the oracle's codes
    assert nan_code_equal(cache.k.cpu().numpy(), orc.st.K)
    assert nan_code_equal(cache.v.cpu().numpy(), orc.st.V)
    for step in range(2):
        so, co, q, outs = orc.step(step)
        _, k, v = wl.step_values(step)
        sg, pg, og = run.step(wl.decode_seqs, q, k, v)
        assert list(sg) == so and [tuple(p) for p in pg] == co
        if step == 0:
            assert len(co) == 1  # the second branch copies the shared tail
        assert nan_code_equal(cache.k.cpu().numpy(), orc.st.K)
        assert nan_code_equal(cache.v.cpu().numpy(), orc.st.V)
        err = max_err(og.cpu().numpy()[0], outs[0])
        assert err <= TOL, err
    assert cache.kv_pool_device_status() == 0


def test_fp8_small_planned_pass():
    wl = synth.workload("fp8_small")
    orc = OracleRun(wl)
    cache, run = make(wl)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    sg, pg, og = run.step(wl.decode_seqs, qh, k, v, planned=True)
    assert list(sg) == so and [tuple(p) for p in pg] == co
    h_plan, _, _ = run.plan(wl.decode_seqs, run.max_blocks(wl.decode_seqs))
    from paged_kv_cache_65_gb300.cache import parse_plan

    plan = parse_plan(h_plan)
    assert plan["kernel"] == 2  # narrow shared segments: the warp-level MMA pass
    assert plan["n_shared_segs"] > 0  # the two branches share 9 blocks
    err = max_err(og.cpu().numpy()[0], orc.attend(0, qh))
    assert err <= TOL, err
    assert cache.kv_pool_device_status() == 0


# block sizes below, at and above the 128-token FP8 stage, and one (192) whose
# blocks the stage covers in 64-row boxes
@pytest.mark.parametrize("G,B", [(1, 16), (2, 8), (4, 32), (8, 64), (8, 16), (4, 128), (2, 192),
                                 (1, 256)])
def test_fp8_ragged_shapes(G, B):
    ctxs = [1, 2, B - 1, B, B + 1, 3 * B + 2, 97, 700]
    wl = fp8_workload("fp8_ragged", G, B, 10 + G + B, ctxs, k_scale=0.25, v_scale=4.0)
    orc = OracleRun(wl)
    cache, run = make(wl)
    so, co, q, outs = orc.step(0)
    _, k, v = wl.step_values(0)
    sg, pg, og = run.step(wl.decode_seqs, q, k, v)
    assert list(sg) == so
    assert nan_code_equal(cache.k.cpu().numpy(), orc.st.K)
    err = max_err(og.cpu().numpy()[0], outs[0])
    assert err <= TOL, (G, B, err)
    assert cache.kv_pool_device_status() == 0


def test_fp8_unused_slots_holding_nan_codes_do_not_leak():
    wl = synth.workload("fp8_small")
    orc = OracleRun(wl)
    cache, run = make(wl, fill=0xFF)  # every unused slot holds the NaN code
    so, co, q, outs = orc.step(0)
    _, k, v = wl.step_values(0)
    _, _, og = run.step(wl.decode_seqs, q, k, v)
    got = og.cpu().numpy()[0]
    assert np.isfinite(got).all()
    assert max_err(got, outs[0]) <= TOL


def test_fp8_qwen_2k_full():
    # every output of all 37 sequences, per sequence and through the plan
    from paged_kv_cache_65_gb300.driver import to_device

    wl = synth.workload("qwen_2k_fp8")
    orc = OracleRun(wl)
    cache, run = make(wl)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    sg, pg, og = run.step(wl.decode_seqs, qh, k, v)
    assert list(sg) == so
    ref = orc.attend(0, qh)
    assert max_err(og.cpu().numpy()[0], ref) <= TOL
    d_table, _, mb = run.tables(wl.decode_seqs)
    h_plan, d_plan, ws = run.plan(wl.decode_seqs, mb)
    got = run.attend_planned(0, to_device(qh, "bf16", "cuda"), d_table, mb, h_plan, d_plan, ws)
    assert max_err(got.cpu().numpy(), ref) <= TOL
    # the pool's written rows are the oracle's codes
    assert nan_code_equal(cache.k.cpu().numpy(), orc.st.K)
    assert nan_code_equal(cache.v.cpu().numpy(), orc.st.V)
    assert cache.kv_pool_device_status() == 0


@pytest.mark.parametrize("pinned,path", [(False, 0), (True, 0), (True, 3)])
def test_fp8_host_buffer_step(pinned, path):
    # the whole-step C entry point with host buffers: bf16 q and new K/V in,
    # quantized on the device, float32 out; pageable buffers go through the
    # staging area, page-locked ones are read and written in place; path 3:
    # the step's planned pass on tcgen05
    wl = synth.workload("fp8_small")
    orc = OracleRun(wl)
    cache, run = make(wl, path=path)
    max_blocks = 32
    n = len(wl.decode_seqs)
    staging = torch.empty(cache.kv_decode_step_staging_bytes(n, wl.n_q_heads, max_blocks),
                          dtype=torch.uint8, device="cuda")
    for step in range(2):
        so, co = orc.reserve_step()
        q = orc.write_step(step, so, co)
        _, k, v = wl.step_values(step)
        if pinned:
            out = torch.zeros((1, n, wl.n_q_heads, wl.head_dim), dtype=torch.float32).pin_memory()
            args = [torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()
                    for a in (q[None], k, v)]
        else:
            out = np.zeros((1, n, wl.n_q_heads, wl.head_dim), dtype=np.float32)
            args = [q[None], k, v]
        cache.kv_decode_step_host(wl.decode_seqs, wl.n_q_heads, max_blocks, *args, out, staging)
        got = out if isinstance(out, np.ndarray) else out.numpy()
        assert max_err(got[0], orc.attend(0, q)) <= TOL
    assert nan_code_equal(cache.k.cpu().numpy(), orc.st.K)
    assert nan_code_equal(cache.v.cpu().numpy(), orc.st.V)
    assert cache.kv_pool_device_status() == 0


def test_fp8_scales_are_checked():
    from paged_kv_cache_65_gb300 import PagedKVCache

    wl = synth.workload("fp8_small")
    cache, _ = make(wl)
    for bad in [(0.0, 1.0), (1.0, -2.0), (float("inf"), 1.0), (float("nan"), 1.0)]:
        with pytest.raises(Exception):
            cache.kv_pool_set_fp8_scales(*bad)
    bf = PagedKVCache(1, 8, 16, 2, 128, "bf16")
    with pytest.raises(Exception):
        bf.kv_pool_set_fp8_scales(1.0, 1.0)


# ---------------------------------------------------------------- tcgen05


def attend_ways(cache, run, wl, qh, paths=(2, 3)):
    """One step's attention per sequence and through the plan, on each pass."""
    from paged_kv_cache_65_gb300 import _lib
    from paged_kv_cache_65_gb300.cache import parse_plan
    from paged_kv_cache_65_gb300.driver import to_device

    d_table, d_lens, mb = run.tables(wl.decode_seqs)
    qd = to_device(qh, "bf16", "cuda")
    outs = {}
    for path in paths:
        cache.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, path)
        outs[("plain", path)] = run.attend(0, qd, d_table, mb, d_lens,
                                           len(wl.decode_seqs)).cpu().numpy()
        h_plan, d_plan, ws_bytes = run.plan(wl.decode_seqs, mb)
        assert parse_plan(h_plan)["kernel"] == path
        outs[("planned", path)] = run.attend_planned(0, qd, d_table, mb, h_plan, d_plan,
                                                     ws_bytes).cpu().numpy()
    return outs


def test_fp8_tc_small_steps_and_planned():
    # two steps on the tcgen05 pass (the first copies the shared tail), then
    # the planned call of a third step
    wl = synth.workload("fp8_small")
    orc = OracleRun(wl)
    cache, run = make(wl, path=3)
    for step in range(2):
        so, co, q, outs = orc.step(step)
        _, k, v = wl.step_values(step)
        sg, pg, og = run.step(wl.decode_seqs, q, k, v)
        assert list(sg) == so and [tuple(p) for p in pg] == co
        assert max_err(og.cpu().numpy()[0], outs[0]) <= TOL
    so, co = orc.reserve_step()
    qh = orc.write_step(2, so, co)
    _, k, v = wl.step_values(2)
    sg, pg = run.reserve(wl.decode_seqs)
    assert list(sg) == so and [tuple(p) for p in pg] == co
    run.write(sg, pg, k, v)
    ref = orc.attend(0, qh)
    for key, got in attend_ways(cache, run, wl, qh).items():
        assert max_err(got, ref) <= TOL, key
    assert nan_code_equal(cache.k.cpu().numpy(), orc.st.K)
    assert nan_code_equal(cache.v.cpu().numpy(), orc.st.V)
    assert cache.kv_pool_device_status() == 0


@pytest.mark.parametrize("G,B", [(1, 16), (2, 8), (4, 32), (8, 64), (8, 16), (4, 128), (2, 192),
                                 (1, 256)])
def test_fp8_tc_ragged_shapes(G, B):
    # stages that end inside a block and inside a 16-row MMA step, plus a
    # prefix forked into branches whose shared segment carries up to 32
    # query columns (its partly filled tail is copied by every branch)
    ctxs = [1, 2, B - 1, B, B + 1, 3 * B + 2, 97, 700]
    ops = [("append", s, c - 1, s) for s, c in enumerate(ctxs) if c > 1]
    n_br = min(8, 32 // G)
    fork = max(3 * B + 5, 300)
    ops += [("append", 100, fork, 99)] + [("fork", 100, 200 + i) for i in range(n_br)]
    seqs = list(range(len(ctxs))) + [200 + i for i in range(n_br)]
    seed = 40 + G + B
    wl = synth.Workload("fp8_tc_ragged", 1, 512, B, 2 * G, 2, 128, "fp8_e4m3", seed,
                        synth.permutation((seed, 9), 512), ops, seqs, k_scale=0.25,
                        v_scale=4.0)
    orc = OracleRun(wl)
    cache, run = make(wl, path=3)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    sg, pg = run.reserve(wl.decode_seqs)
    assert list(sg) == so and [tuple(p) for p in pg] == co
    run.write(sg, pg, k, v)
    ref = orc.attend(0, qh)
    for key, got in attend_ways(cache, run, wl, qh, paths=(3,)).items():
        assert max_err(got, ref) <= TOL, (G, B, key)
    assert nan_code_equal(cache.k.cpu().numpy(), orc.st.K)
    assert cache.kv_pool_device_status() == 0


def test_fp8_tc_unused_slots_holding_nan_codes_do_not_leak():
    wl = synth.workload("fp8_small")
    orc = OracleRun(wl)
    cache, run = make(wl, fill=0xFF, path=3)
    so, co, q, outs = orc.step(0)
    _, k, v = wl.step_values(0)
    _, _, og = run.step(wl.decode_seqs, q, k, v)
    got = og.cpu().numpy()[0]
    assert np.isfinite(got).all()
    assert max_err(got, outs[0]) <= TOL


def test_fp8_gqa70b_32k_full_both_passes():
    # all 48 branches, two steps (the first copies 48 shared tails), four
    # ways; the automatic plan takes the tcgen05 pass
    from paged_kv_cache_65_gb300 import _lib
    from paged_kv_cache_65_gb300.cache import parse_plan

    wl = synth.workload("gqa70b_32k_fp8")
    orc = OracleRun(wl)
    cache, run = make(wl)
    for step in range(2):
        so, co = orc.reserve_step()
        qh = orc.write_step(step, so, co)
        _, k, v = wl.step_values(step)
        sg, pg = run.reserve(wl.decode_seqs)
        assert list(sg) == so and [tuple(p) for p in pg] == co
        assert len(co) == (48 if step == 0 else 0)
        run.write(sg, pg, k, v)
        if step == 0:
            cache.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, 0)
            h_auto, _, _ = run.plan(wl.decode_seqs, run.max_blocks(wl.decode_seqs))
            assert parse_plan(h_auto)["kernel"] == 3
        ref = orc.attend(0, qh)
        for key, got in attend_ways(cache, run, wl, qh).items():
            assert max_err(got, ref) <= TOL, (step, key)
    assert nan_code_equal(cache.k.cpu().numpy(), orc.st.K)
    assert nan_code_equal(cache.v.cpu().numpy(), orc.st.V)
    assert cache.kv_pool_device_status() == 0


def test_fp8_shared_8k_full_both_passes():
    # all 16 sequences over the 6144-token shared prefix, four ways
    wl = synth.workload("shared_8k_fp8")
    orc = OracleRun(wl)
    cache, run = make(wl)
    so, co = orc.reserve_step()
    qh = orc.write_step(0, so, co)
    _, k, v = wl.step_values(0)
    sg, pg = run.reserve(wl.decode_seqs)
    assert list(sg) == so and len(pg) == 0
    run.write(sg, pg, k, v)
    ref = orc.attend(0, qh)
    for key, got in attend_ways(cache, run, wl, qh).items():
        assert max_err(got, ref) <= TOL, key
    assert nan_code_equal(cache.k.cpu().numpy(), orc.st.K)
    assert cache.kv_pool_device_status() == 0
