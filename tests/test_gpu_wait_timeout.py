"""Bounded waits on the GPU: a wait that nothing completes gives up after its
limit, the status word reports KV_DEV_WAIT_TIMEOUT, and the device stays
usable (a decode step right after matches the oracle).  The wait is made to
run out with a barrier that nothing arrives on, never with a fault."""

import time

import numpy as np
import pytest

import synth
from oracle.runner import OracleRun

torch = pytest.importorskip("torch")
pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]


def test_wait_gives_up_reports_and_the_device_stays_usable():
    from paged_kv_cache_65_gb300 import PagedKVCache, _lib
    from paged_kv_cache_65_gb300.driver import DeviceRun

    wl = synth.workload("tiny")
    cache = PagedKVCache(wl.n_layers, wl.n_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim,
                         wl.dtype, free_order=wl.free_order)
    cache.k.zero_()
    cache.v.zero_()
    assert cache.kv_pool_device_status() == 0
    for limit_us in (2000, 20000):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        cache.kv_device_wait_selftest(limit_us)
        bits = cache.kv_pool_device_status()  # synchronises
        dt = time.perf_counter() - t0
        assert bits == _lib.KV_DEV_WAIT_TIMEOUT
        assert limit_us * 1e-6 <= dt < limit_us * 1e-6 + 1.0, dt
    assert cache.kv_pool_device_status() == 0  # reading cleared it
    with pytest.raises(Exception):
        cache.kv_device_wait_selftest(0)
    # the same context runs a decode step that matches the oracle
    orc = OracleRun(wl)
    run = DeviceRun(cache, wl.n_q_heads)
    for op in wl.build_ops:
        run.apply(op, wl.append_values)
    so, co, q, outs = orc.step(0)
    _, k, v = wl.step_values(0)
    sg, _, og = run.step(wl.decode_seqs, q, k, v)
    assert list(sg) == so
    assert float(np.max(np.abs(og.cpu().numpy()[0].astype(np.float64) - outs[0]))) <= 1e-5
    assert cache.kv_pool_device_status() == 0
