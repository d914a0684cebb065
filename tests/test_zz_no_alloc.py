"""The no-allocation decode entry point, for callers that cannot allocate
device memory (under an allocator that already owns all device memory, or
with no allocator at all).

Its workspace is the library's static scratch array and it runs the same
kernels as the entry point that takes a caller workspace, so on two calls in
a row that reuse the same array its outputs must be bit-identical to that
entry point's, and within the tolerance of the oracle's attention.  This file
is collected last so that a failure here cannot hide the other GPU tests.
"""

import numpy as np
import pytest

import synth
from oracle.runner import OracleRun

torch = pytest.importorskip("torch")
pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]

TOL = {"f32": 1e-5, "bf16": 2e-3}


def build(dtype, D, G, B, lens, seed):
    from paged_kv_cache_65_gb300 import PagedKVCache
    from paged_kv_cache_65_gb300.driver import DeviceRun

    n_blocks = sum(-(-l // B) for l in lens) + len(lens) + 3
    ops = [("append", s, l - 1, s) for s, l in enumerate(lens) if l > 1]
    wl = synth.Workload("noalloc", 1, n_blocks, B, 2 * G, 2, D, dtype, seed,
                        synth.permutation((seed, 9), n_blocks), ops, list(range(len(lens))))
    cache = PagedKVCache(1, n_blocks, B, 2, D, dtype, free_order=wl.free_order)
    cache.k.zero_()
    cache.v.zero_()
    run = DeviceRun(cache, wl.n_q_heads)
    for op in wl.build_ops:
        run.apply(op, wl.append_values)
    q, k, v = wl.step_values(0)
    run.write(*run.reserve(wl.decode_seqs), k, v)
    orc = OracleRun(wl)
    orc.write_step(0, *orc.reserve_step())
    return wl, cache, run, orc


@pytest.mark.parametrize("dtype,D,G,B", [("bf16", 128, 4, 16), ("f32", 64, 4, 4)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(dtype, D, G, B):
    from paged_kv_cache_65_gb300.driver import to_device

    lens = [1, 17, 300, 2049, 45]
    wl, cache, run, orc = build(dtype, D, G, B, lens, seed=21)
    d_table, d_lens, mb = run.tables(wl.decode_seqs)
    n = len(lens)
    for call in range(2):  # the second call reuses the array the first one left behind
        q = synth.storage_values(synth.normal_f32((99, call), (n, wl.n_q_heads, D)), dtype)
        qd = to_device(q, dtype, "cuda")
        ref = run.attend(0, qd, d_table, mb, d_lens, n)
        got = torch.full_like(ref, float("nan"))
        cache.paged_decode_attention_noalloc(0, qd, wl.n_q_heads, d_table, mb, d_lens, n, got)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)  # same kernels, same inputs: same bits
        err = float(np.max(np.abs(got.cpu().numpy().astype(np.float64) - orc.attend(0, q))))
        assert err <= TOL[dtype], err
    assert cache.kv_pool_device_status() == 0


def test_noalloc_rejects_requests_beyond_the_scratch_size():
    from paged_kv_cache_65_gb300 import KVError
    from paged_kv_cache_65_gb300 import _lib

    wl, cache, run, _ = build("bf16", 128, 4, 16, [5, 9], seed=3)
    n_seq = 5000  # its workspace would be far above the 16 MiB array
    assert cache.paged_decode_workspace_bytes(n_seq, wl.n_q_heads) > 16 << 20
    d_table, d_lens, mb = run.tables(wl.decode_seqs)
    out = torch.empty((2, wl.n_q_heads, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(KVError) as e:
        cache.paged_decode_attention_noalloc(0, out, wl.n_q_heads, d_table, mb, d_lens, n_seq, out)
    assert e.value.status == _lib.KV_ERR_SCRATCH_TOO_SMALL
