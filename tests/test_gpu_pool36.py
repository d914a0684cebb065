"""Full-size serving step (36 Qwen3-8B-shaped layers, 128 lognormal
sequences, 25 % sharing a 6144-token prefix, B = 16) in the launch
configuration the benchmark times (planned tensor-core pass), checked on
sampled outputs: the sampled sequences' history rows are read back from the
pool before the step (the pool is filled by torch's generator, not by this
library), the new token and q come from a seeded host generator, and the
oracle attends over the contiguous rows."""

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


def test_pool36_sampled_parity():
    import bench
    from paged_kv_cache_65_gb300.driver import to_device, to_host_bits

    if torch.cuda.get_device_properties(0).total_memory < 200e9:
        pytest.skip("needs a GPU with more than 200 GB")
    wl, cache, run = bench.setup("pool36", 16, "cuda")
    seqs = wl.decode_seqs
    sample, layers = [0, 31, 40, 127], [0, 35]
    B = cache.B
    hist = {}
    for i in sample:
        s = seqs[i]
        table, lens = cache.seq_block_table([s], run.max_blocks([s]))
        n = int(lens[0])
        rows = torch.from_numpy(table[0, : -(-n // B)].astype(np.int64)).cuda()
        for layer in layers:
            k = cache.k[layer].index_select(0, rows).reshape(-1, cache.H, cache.D)[:n]
            v = cache.v[layer].index_select(0, rows).reshape(-1, cache.H, cache.D)[:n]
            hist[(i, layer)] = (to_host_bits(k), to_host_bits(v))
    n_seq = len(seqs)
    q = synth.storage_values(synth.normal_f32((44, 0), (n_seq, wl.n_q_heads, wl.head_dim)), "bf16")
    kv = synth.storage_values(synth.normal_f32((44, 1), (wl.n_layers, n_seq, 2, wl.n_kv_heads,
                                                          wl.head_dim)), "bf16")
    k_new, v_new = np.ascontiguousarray(kv[:, :, 0]), np.ascontiguousarray(kv[:, :, 1])
    slots, pairs = run.reserve(seqs)
    run.write(slots, pairs, k_new, v_new)
    d_table, d_lens, mb = run.tables(seqs)
    h_plan, d_plan, ws_bytes = run.plan(seqs, mb)
    qd = to_device(q, "bf16", "cuda")
    for layer in layers:
        out = run.attend_planned(layer, qd, d_table, mb, h_plan, d_plan, ws_bytes).cpu().numpy()
        for i in sample:
            kh, vh = hist[(i, layer)]
            K = np.concatenate([to_f64(kh, "bf16"), to_f64(k_new[layer, i:i + 1], "bf16")])
            V = np.concatenate([to_f64(vh, "bf16"), to_f64(v_new[layer, i:i + 1], "bf16")])
            ref = decode_attention(to_f64(q[i], "bf16"), K, V)
            assert float(np.max(np.abs(out[i] - ref))) <= 2e-3, (i, layer)
    assert cache.kv_pool_device_status() == 0
