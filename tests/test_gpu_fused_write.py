"""The planned split pass with the step's slot write fused in
(`paged_decode_partials_planned_write`): each listed sequence's newest token
is written by the CTA that reads the block it lands in, just before that
read.  The pools must be byte-identical to the oracle's after every step
(its slot writes and copy-on-write copies), and the outputs within the
tolerance of the oracle's attention, on both tensor-core passes, with
copy-on-write steps, FP8 pools and several layers."""

import numpy as np
import pytest

import synth
from oracle.runner import OracleRun

torch = pytest.importorskip("torch")
pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]

TOL = 2e-3


def make(wl, path):
    from paged_kv_cache_65_gb300 import PagedKVCache, _lib
    from paged_kv_cache_65_gb300.driver import DeviceRun

    cache = PagedKVCache(wl.n_layers, wl.n_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim,
                         wl.dtype, free_order=wl.free_order)
    if wl.dtype == "fp8_e4m3":
        cache.kv_pool_set_fp8_scales(wl.k_scale, wl.v_scale)
    cache.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, path)
    cache.k.zero_()
    cache.v.zero_()
    run = DeviceRun(cache, wl.n_q_heads)
    for op in wl.build_ops:
        run.apply(op, wl.append_values)
    return cache, run


def same_pool(gpu, ref, fp8):
    from paged_kv_cache_65_gb300.driver import to_host_bits

    a = to_host_bits(gpu)
    if not fp8:
        return np.array_equal(a, ref)
    na, nb = (a & 0x7F) == 0x7F, (ref & 0x7F) == 0x7F  # any two NaN codes match
    return bool(np.array_equal(na, nb) and np.array_equal(a[~na], ref[~nb]))


def fused_steps(wl, path, steps, expect_cow=None):
    from paged_kv_cache_65_gb300.driver import to_device

    orc = OracleRun(wl)
    cache, run = make(wl, path)
    seqs = wl.decode_seqs
    fp8 = wl.dtype == "fp8_e4m3"
    for step in range(steps):
        so, co = orc.reserve_step()
        qh = orc.write_step(step, so, co)
        _, k, v = wl.step_values(step)
        slots, pairs = run.reserve(seqs)
        assert list(slots) == so and [tuple(p) for p in pairs] == co
        if expect_cow is not None:
            assert len(co) == expect_cow[step]
        if len(pairs):
            cache.cow_copy(torch.from_numpy(np.ascontiguousarray(pairs)).cuda(), len(pairs))
        d_table, _, mb = run.tables(seqs)
        h_plan, d_plan, ws_bytes = run.plan(seqs, mb)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        qd = to_device(qh, "bf16", "cuda")
        kd, vd = to_device(k, "bf16", "cuda"), to_device(v, "bf16", "cuda")
        for layer in range(wl.n_layers):
            ql = qd[layer] if qd.dim() == 4 else qd
            out = torch.empty((len(seqs), wl.n_q_heads, wl.head_dim), dtype=torch.float32,
                              device="cuda")
            cache.paged_decode_partials_planned_write(layer, ql, wl.n_q_heads, kd[layer],
                                                      vd[layer], d_table, mb, d_plan, h_plan,
                                                      ws)
            cache.paged_decode_merge_planned(wl.n_q_heads, d_plan, h_plan, out, ws)
            qo = qh[layer] if qh.ndim == 4 else qh
            ref = orc.attend(layer, qo)
            err = float(np.max(np.abs(out.cpu().numpy().astype(np.float64) - ref)))
            assert err <= TOL, (step, layer, err)
        torch.cuda.synchronize()
        assert same_pool(cache.k, orc.st.K, fp8), step
        assert same_pool(cache.v, orc.st.V, fp8), step
    assert cache.kv_pool_device_status() == 0


@pytest.mark.parametrize("path", [2, 3])
def test_fused_write_qwen_2k(path):
    fused_steps(synth.workload("qwen_2k"), path, 2)


@pytest.mark.parametrize("path", [2, 3])
def test_fused_write_shared_8k(path):
    fused_steps(synth.workload("shared_8k"), path, 2)


@pytest.mark.parametrize("path", [0, 2])
def test_fused_write_gqa70b_32k_with_copy_on_write(path):
    # the first step copies 48 shared tails, then each branch's new token
    # goes into its copy (automatic choice: tcgen05)
    fused_steps(synth.workload("gqa70b_32k"), path, 2, expect_cow=[48, 0])


@pytest.mark.parametrize("path", [0, 3])
def test_fused_write_fp8_pool(path):
    # quantized on the way in, one copy-on-write in the first step; the
    # warp-level pass (automatic) and tcgen05
    fused_steps(synth.workload("fp8_small"), path, 3, expect_cow=[1, 0, 0])


def test_fused_write_fp8_gqa70b_32k_with_copy_on_write():
    # FP8 codes written by the tcgen05 producers (automatic choice) after 48
    # copy-on-write copies of shared tails
    fused_steps(synth.workload("gqa70b_32k_fp8"), 0, 2, expect_cow=[48, 0])


@pytest.mark.parametrize("B,path", [(8, 2), (16, 3), (32, 2), (64, 3)])
def test_fused_write_several_layers_and_forks(B, path):
    # three layers; sequences forked from a prefix whose tail block is partly
    # filled (the parent stays alive, so every branch copies it), a lone
    # sequence at a block boundary, and short ones
    G, H, L = 4, 2, 3
    ops = [("append", 100, 3 * B + 3, 0), ("fork", 100, 0), ("fork", 100, 1), ("fork", 100, 2),
           ("append", 3, 5 * B - 1, 3), ("append", 4, 1, 4), ("append", 1, 7, 5)]
    wl = synth.Workload("fused", L, 256, B, H * G, H, 128, "bf16", 60 + B,
                        synth.permutation((60 + B, 3), 256), ops, [0, 1, 2, 3, 4, 5])
    fused_steps(wl, path, 3)
