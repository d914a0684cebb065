"""GPU parity of the chunked-prefill attention (through the C ABI) with the
oracle on the same seeded inputs: bfloat16 K/V, float32 accumulation,
max-abs error within 2e-3."""

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


def make(wl, fill_nan=False):
    from paged_kv_cache_65_gb300 import PagedKVCache
    from paged_kv_cache_65_gb300.driver import DeviceRun

    cache = PagedKVCache(wl.n_layers, wl.n_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim,
                         wl.dtype, free_order=wl.free_order)
    if fill_nan:
        cache.k.fill_(float("nan"))
        cache.v.fill_(float("nan"))
    else:
        cache.k.zero_()
        cache.v.zero_()
    run = DeviceRun(cache, wl.n_q_heads)
    for op in wl.build_ops:
        run.apply(op, wl.append_values)
    return cache, run


def check_against_oracle(wl, fill_nan=False, chunk_index=None, out_dtype=None, scheduled=False):
    """Largest error of the chunks' outputs against the oracle.  With bf16
    outputs the error is taken after removing half a bf16 ulp of the exact
    value (2^-8 relative): a row that sees few keys can have |out| ~ 4."""
    orc = OracleRun(wl)
    cache, run = make(wl, fill_nan)
    _, _, q = orc.prefill_step(0)
    q2, k, v = wl.chunk_values(0)
    assert np.array_equal(q, q2)
    og = run.prefill_step(wl.chunks, q, k, v, out_dtype=out_dtype, scheduled=scheduled)
    got = og.float().cpu().numpy()[0]
    ref = orc.prefill_attend(0, q, chunk_index)
    offs = np.cumsum([0] + [c for _, c in wl.chunks])
    worst = 0.0
    for i, r in ref.items():
        g = got[offs[i]:offs[i] + wl.chunks[i][1]]
        assert np.isfinite(g).all()
        err = np.abs(g - r)
        if out_dtype is not None:
            err = np.maximum(err - 2.0 ** -8 * np.abs(r), 0.0)
        worst = max(worst, float(np.max(err)) if r.size else 0.0)
    assert cache.kv_pool_device_status() == 0
    return worst


def test_prefill_tiny_all_rows():
    assert check_against_oracle(synth.workload("prefill_tiny")) <= TOL


def test_prefill_4k_round_against_oracle():
    # every row of the 8 chunks of 512 tokens after histories 0 .. 7680
    # (4096 query rows), natural grid
    assert check_against_oracle(synth.workload("prefill_4k")) <= TOL


def ragged(G, B, hist, chunks, seed):
    n_blocks = sum(-(-(h + c) // B) for h, c in zip(hist, chunks)) + len(hist) + 4
    ops = [("append", s, h, s) for s, h in enumerate(hist) if h > 0]
    return synth.PrefillWorkload("ragged_prefill", 1, n_blocks, B, 2 * G, 2, 128, "bf16", seed,
                                 synth.permutation((seed, 1), n_blocks), ops,
                                 list(range(len(hist))), "", list(enumerate(chunks)))


@pytest.mark.parametrize("G,B", [(1, 16), (2, 8), (4, 32), (8, 64), (4, 16)])
def test_prefill_ragged_shapes(G, B):
    hist = [0, 5, 130, 1000, 17]
    chunks = [1, 17, 300, 64, 129]
    assert check_against_oracle(ragged(G, B, hist, chunks, seed=G * 100 + B)) <= TOL


def test_prefill_unused_slots_holding_nan_do_not_leak():
    wl = ragged(4, 16, [3, 0, 40], [9, 33, 100], seed=7)
    assert check_against_oracle(wl, fill_nan=True) <= TOL


def test_prefill_bf16_output():
    wl = ragged(4, 16, [0, 200], [70, 31], seed=8)
    assert check_against_oracle(wl, out_dtype=torch.bfloat16) <= TOL


def test_prefill_in_chunks_equals_one_pass():
    # "KV 缓存管理": chunked prefill is equivalent to one pass; on the device
    # a 300-token prompt in chunks of 128 matches the same prompt at once
    from paged_kv_cache_65_gb300.driver import to_host_bits  # noqa: F401

    G, B, S = 4, 16, 300
    wl1 = ragged(G, B, [0], [S], seed=11)
    q, k, v = wl1.chunk_values(0)
    cache, run = make(wl1)
    whole = run.prefill_step([(0, S)], q, k, v).cpu().numpy()[0]
    cache2, run2 = make(wl1)
    parts = []
    for a in range(0, S, 128):
        b = min(S, a + 128)
        parts.append(run2.prefill_step([(0, b - a)], q[a:b], k[:, a:b], v[:, a:b]).cpu().numpy()[0])
    assert float(np.max(np.abs(np.concatenate(parts) - whole))) <= 1e-3


def test_prefill_chunk_longer_than_max_chunk_is_flagged():
    wl = ragged(4, 16, [0], [200], seed=12)
    cache, run = make(wl)
    q, k, v = wl.chunk_values(0)
    run.prefill_step(wl.chunks, q, k, v, max_chunk=100)
    assert cache.kv_pool_device_status() & 16
    assert cache.kv_pool_device_status() == 0


# ------------------------------------------------- heaviest-first work order
def test_prefill_4k_scheduled_against_oracle():
    # every row, in the bench's heaviest-first launch order
    assert check_against_oracle(synth.workload("prefill_4k"), scheduled=True) <= TOL


@pytest.mark.parametrize("G,B", [(1, 16), (2, 8), (8, 64), (4, 16)])
def test_prefill_scheduled_ragged_against_oracle(G, B):
    hist = [0, 5, 130, 1000, 17]
    chunks = [1, 17, 300, 64, 129]
    assert check_against_oracle(ragged(G, B, hist, chunks, seed=G * 100 + B + 1),
                                scheduled=True) <= TOL


@pytest.mark.parametrize("name", ["prefill_4k", "ragged"])
def test_prefill_scheduled_equals_natural_grid_bit_for_bit(name):
    # a CTA computes the same rows with the same arithmetic whichever order
    # launches it: the outputs are identical, not merely close
    wl = synth.workload(name) if name != "ragged" else ragged(4, 16, [0, 900, 33], [250, 7, 128],
                                                             seed=21)
    q, k, v = wl.chunk_values(0)
    outs = []
    for scheduled in (False, True):
        cache, run = make(wl)
        outs.append(run.prefill_step(wl.chunks, q, k, v, scheduled=scheduled).cpu().numpy())
        assert cache.kv_pool_device_status() == 0
    assert np.array_equal(outs[0], outs[1])


def test_prefill_schedule_for_other_chunk_lengths_is_flagged():
    # an order built for a 150-token chunk, given a 200-token chunk: that
    # sequence is skipped and flagged, the other one still computed
    from paged_kv_cache_65_gb300.driver import to_device

    wl = ragged(4, 16, [0, 40], [200, 64], seed=13)
    cache, run = make(wl)
    q, k, v = wl.chunk_values(0)
    ref = run.prefill_step(wl.chunks, q, k, v).cpu().numpy()[0]
    assert cache.kv_pool_device_status() == 0
    d_table, d_lens, mb = run.tables([0, 1])
    lens = d_lens.cpu().numpy()
    starts = np.array([0, 200, 264], dtype=np.int32)
    planned = np.array([0, 150, 214], dtype=np.int32)
    sched = cache.paged_prefill_schedule(planned, lens, wl.n_q_heads)
    d_sched = torch.from_numpy(sched).to("cuda")
    qd = to_device(q, cache.dtype, torch.device("cuda"))
    out = torch.full((264, wl.n_q_heads, wl.head_dim), 7.0, device="cuda")
    cache.paged_prefill_attention_scheduled(0, qd, wl.n_q_heads, d_table, mb,
                                            torch.from_numpy(starts).to("cuda"), d_lens, 2,
                                            d_sched, len(sched), out, 0.0, run.stream)
    got = out.cpu().numpy()
    assert cache.kv_pool_device_status() & 16
    assert cache.kv_pool_device_status() == 0
    assert (got[:200] == 7.0).all()  # skipped
    assert np.array_equal(got[200:], ref[200:])


# ------------------------------------------------------------ FP8 pools
# paged_prefill_attention_staged: an FP8 (E4M3) pool is read through an exact
# bfloat16 copy of the blocks each chunk's sequence reads; the outputs are
# attention over the pool's dequantized values, which is what the oracle's
# FP8 store gathers.

def fp8_prefill(G, B, hist, chunks, seed, k_scale=0.5, v_scale=2.0, H=2, n_blocks=None):
    n_blocks = n_blocks or sum(-(-(h + c) // B) for h, c in zip(hist, chunks)) + len(hist) + 4
    ops = [("append", s, h, s) for s, h in enumerate(hist) if h > 0]
    return synth.PrefillWorkload("fp8_prefill", 1, n_blocks, B, H * G, H, 128, "fp8_e4m3", seed,
                                 synth.permutation((seed, 1), n_blocks), ops,
                                 list(range(len(hist))), "", list(enumerate(chunks)),
                                 k_scale=k_scale, v_scale=v_scale)


def make_fp8(wl, fill=0):
    from paged_kv_cache_65_gb300 import PagedKVCache
    from paged_kv_cache_65_gb300.driver import DeviceRun

    cache = PagedKVCache(wl.n_layers, wl.n_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim,
                         wl.dtype, free_order=wl.free_order)
    cache.kv_pool_set_fp8_scales(wl.k_scale, wl.v_scale)
    cache.k.fill_(fill)
    cache.v.fill_(fill)
    run = DeviceRun(cache, wl.n_q_heads)
    for op in wl.build_ops:
        run.apply(op, wl.append_values)
    return cache, run


def fp8_round(wl, fill=0, scheduled=False):
    """Outputs of one FP8 prefill round and the oracle's, per chunk."""
    orc = OracleRun(wl)
    cache, run = make_fp8(wl, fill)
    _, _, q = orc.prefill_step(0)
    _, k, v = wl.chunk_values(0)
    og = run.prefill_step(wl.chunks, q, k, v, scheduled=scheduled)
    got = og.float().cpu().numpy()[0]
    ref = orc.prefill_attend(0, q)
    assert cache.kv_pool_device_status() == 0
    return cache, got, ref


def fp8_worst(wl, got, ref):
    offs = np.cumsum([0] + [c for _, c in wl.chunks])
    worst = 0.0
    for i, r in ref.items():
        g = got[offs[i]:offs[i] + wl.chunks[i][1]]
        assert np.isfinite(g).all()
        worst = max(worst, float(np.max(np.abs(g - r))) if r.size else 0.0)
    return worst


def test_prefill_fp8_tiny_all_rows():
    wl = synth.workload("prefill_tiny")
    import dataclasses

    wl = dataclasses.replace(wl, dtype="fp8_e4m3", k_scale=0.25, v_scale=4.0)
    _, got, ref = fp8_round(wl)
    assert fp8_worst(wl, got, ref) <= TOL


@pytest.mark.parametrize("G,B", [(1, 16), (2, 8), (4, 32), (8, 64), (2, 32)])
def test_prefill_fp8_ragged_shapes(G, B):
    # chunks starting and ending inside blocks, a chunk of one token, a
    # sequence with no history; unused slots hold NaN codes (0xFF)
    wl = fp8_prefill(G, B, [0, 5, B - 1, 3 * B + 7], [1, B + 3, 2 * B, 130], 40 + G + B)
    _, got, ref = fp8_round(wl, fill=0xFF)
    assert fp8_worst(wl, got, ref) <= TOL


def test_prefill_fp8_scheduled_matches_natural():
    wl = fp8_prefill(4, 16, [0, 300, 1000, 70], [200, 33, 128, 400], 51)
    _, nat, ref = fp8_round(wl)
    _, sch, _ = fp8_round(wl, scheduled=True)
    assert np.array_equal(nat, sch)
    assert fp8_worst(wl, nat, ref) <= TOL


def test_prefill_fp8_4k_round():
    # the 4096-token round (8 chunks of 512 after histories 0 .. 7680) over an
    # FP8 pool, every row against the oracle
    import dataclasses

    wl = dataclasses.replace(synth.workload("prefill_4k"), dtype="fp8_e4m3", k_scale=0.5,
                             v_scale=1.0)
    _, got, ref = fp8_round(wl, scheduled=True)
    assert fp8_worst(wl, got, ref) <= TOL


def test_prefill_staged_bf16_pool_reads_in_place():
    # a bfloat16 pool needs no workspace and gives the plain call's bits
    import torch as T

    from paged_kv_cache_65_gb300 import _lib

    wl = ragged(4, 16, [0, 37, 200], [45, 130, 1], 61)
    cache, run = make(wl)
    orc = OracleRun(wl)
    _, _, q = orc.prefill_step(0)
    _, k, v = wl.chunk_values(0)
    plain = run.prefill_step(wl.chunks, q, k, v)[0]
    assert cache.paged_prefill_staging_bytes(3, 64) == 0
    from paged_kv_cache_65_gb300.driver import to_device

    seqs = [s for s, _ in wl.chunks]
    d_table, d_lens, mb = run.tables(seqs)
    starts = np.zeros(len(wl.chunks) + 1, dtype=np.int32)
    starts[1:] = np.cumsum([n for _, n in wl.chunks])
    out = T.zeros_like(plain)
    cache.paged_prefill_attention_staged(0, to_device(q, "bf16", "cuda"), wl.n_q_heads, d_table,
                                         mb, T.from_numpy(starts).cuda(), d_lens, len(seqs), out,
                                         None, max_chunk=int(max(n for _, n in wl.chunks)))
    T.cuda.synchronize()
    assert T.equal(out, plain)
    assert _lib.KV_OK == 0


def test_prefill_fp8_bad_table_entry_is_flagged_not_read():
    # an out-of-range block id in a table: flagged, its copy zeroed, no read
    # outside the pool, the other rows unchanged in kind (finite)
    import torch as T

    from paged_kv_cache_65_gb300 import _lib
    from paged_kv_cache_65_gb300.driver import to_device

    wl = fp8_prefill(4, 16, [40, 0], [20, 17], 77)
    cache, run = make_fp8(wl)
    orc = OracleRun(wl)
    _, _, q = orc.prefill_step(0)
    _, k, v = wl.chunk_values(0)
    run.prefill_step(wl.chunks, q, k, v)
    assert cache.kv_pool_device_status() == 0
    seqs = [s for s, _ in wl.chunks]
    d_table, d_lens, mb = run.tables(seqs)
    d_table[0, 1] = wl.n_blocks + 9
    starts = np.zeros(len(wl.chunks) + 1, dtype=np.int32)
    starts[1:] = np.cumsum([n for _, n in wl.chunks])
    ws = T.empty(cache.paged_prefill_staging_bytes(len(seqs), mb), dtype=T.uint8, device="cuda")
    out = T.zeros((int(starts[-1]), wl.n_q_heads, 128), dtype=T.float32, device="cuda")
    cache.paged_prefill_attention_staged(0, to_device(q, "bf16", "cuda"), wl.n_q_heads, d_table,
                                         mb, T.from_numpy(starts).cuda(), d_lens, len(seqs), out,
                                         ws, max_chunk=20)
    T.cuda.synchronize()
    assert cache.kv_pool_device_status() & _lib.KV_DEV_BAD_BLOCK_ID
    assert T.isfinite(out).all()
