"""Full-size serving step (36 Qwen3-8B-shaped layers, 128 lognormal
sequences, 25 % sharing a 6144-token prefix) at block sizes 8, 16 and 32,
in the launch configuration the benchmark times (sharing-aware plan,
automatic kernel choice), checked on every output of every sequence in
layers 0, 17 and 35.

The history is the pool's content as torch's device generator filled it
(this library writes none of it): each sequence's history rows of the
checked layers are copied aside with torch before the step.  The new token
and q come from a seeded host generator; the oracle attends over the
contiguous rows plus the new token."""

import numpy as np
import pytest

import synth
from oracle.attention import decode_attention
from oracle.kv_store import to_f64

torch = pytest.importorskip("torch")
pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]

LAYERS = (0, 17, 35)


@pytest.mark.parametrize("block_size", [8, 16, 32])
def test_pool36_full_parity(block_size):
    import bench
    from paged_kv_cache_65_gb300.driver import to_device, to_host_bits

    if torch.cuda.get_device_properties(0).total_memory < 200e9:
        pytest.skip("needs a GPU with more than 200 GB")
    try:
        wl, cache, run = bench.setup("pool36", block_size, "cuda")
        seqs = wl.decode_seqs
        B = cache.B
        hist = {}
        for i, s in enumerate(seqs):
            table, lens = cache.seq_block_table([s], run.max_blocks([s]))
            n = int(lens[0])
            rows = torch.from_numpy(table[0, : -(-n // B)].astype(np.int64)).cuda()
            for layer in LAYERS:
                k = cache.k[layer].index_select(0, rows).reshape(-1, cache.H, cache.D)[:n]
                v = cache.v[layer].index_select(0, rows).reshape(-1, cache.H, cache.D)[:n]
                hist[(i, layer)] = (k.clone(), v.clone())
        n_seq = len(seqs)
        q = synth.storage_values(synth.normal_f32((44, 0), (n_seq, wl.n_q_heads, wl.head_dim)),
                                 "bf16")
        kv = synth.storage_values(synth.normal_f32((44, 1), (wl.n_layers, n_seq, 2,
                                                              wl.n_kv_heads, wl.head_dim)),
                                  "bf16")
        k_new, v_new = np.ascontiguousarray(kv[:, :, 0]), np.ascontiguousarray(kv[:, :, 1])
        slots, pairs = run.reserve(seqs)
        assert len(pairs) == 0  # the shared prefix is whole blocks at every block size
        run.write(slots, pairs, k_new, v_new)
        d_table, d_lens, mb = run.tables(seqs)
        h_plan, d_plan, ws_bytes = run.plan(seqs, mb)
        qd = to_device(q, "bf16", "cuda")
        worst = 0.0
        for layer in LAYERS:
            out = run.attend_planned(layer, qd, d_table, mb, h_plan, d_plan,
                                     ws_bytes).cpu().numpy()
            for i in range(n_seq):
                kh, vh = (to_host_bits(t) for t in hist.pop((i, layer)))
                K = np.concatenate([to_f64(kh, "bf16"), to_f64(k_new[layer, i:i + 1], "bf16")])
                V = np.concatenate([to_f64(vh, "bf16"), to_f64(v_new[layer, i:i + 1], "bf16")])
                ref = decode_attention(to_f64(q[i], "bf16"), K, V)
                err = float(np.max(np.abs(out[i] - ref)))
                assert err <= 2e-3, (block_size, layer, i, err)
                worst = max(worst, err)
        assert cache.kv_pool_device_status() == 0
        print(f"pool36 B={block_size}: {n_seq} sequences x {len(LAYERS)} layers, "
              f"max abs error {worst:.2e}")
    finally:
        hist = None
        wl = cache = run = None
        import gc

        gc.collect()
        torch.cuda.empty_cache()
