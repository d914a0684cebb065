"""Prefix cache through the device path: requests that reuse cached full
blocks ("KV 缓存管理", radix-tree section: longest prefix match, block-aligned
truncation ``S_usable = floor(S_match / B) * B``, leaf-first LRU eviction)
run their slot writes, copy-on-write copies and decode steps on the GPU, and
the same request stream runs through the oracle's prefix cache, K/V store
and attention.  Slots, copy pairs and match lengths are bit-exact, the pools
are byte-identical after every stage, and the attention outputs (plain and
sharing-aware passes, both tensor-core kernels) are within 2e-3."""

import numpy as np
import pytest

import synth
from oracle.attention import decode_attention
from oracle.kv_store import KVStore, to_f64
from oracle.prefix_cache import PrefixCachingBlockManager

torch = pytest.importorskip("torch")
pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]

TOL = 2e-3
N, B, HQ, HKV, D = 48, 16, 8, 2, 128
SALT = 0x5EED5A17
SEED = 65


class Pair:
    """The oracle and the library fed the same calls and values."""

    def __init__(self):
        from paged_kv_cache_65_gb300 import PagedKVCache
        from paged_kv_cache_65_gb300.driver import DeviceRun

        order = synth.permutation((SEED, 0), N)
        self.orc = PrefixCachingBlockManager(N, B, order, salt=SALT)
        self.st = KVStore(1, N, B, HKV, D, "bf16")
        self.c = PagedKVCache(1, N, B, HKV, D, "bf16", free_order=order)
        self.c.k.zero_()
        self.c.v.zero_()
        self.c.kv_prefix_cache_enable(SALT)
        self.run = DeviceRun(self.c, HQ)
        self.calls = 0

    def values(self, n):
        self.calls += 1
        x = synth.storage_values(synth.normal_f32((SEED, 1, self.calls), (1, n, 2, HKV, D)),
                                 "bf16")
        return np.ascontiguousarray(x[:, :, 0]), np.ascontiguousarray(x[:, :, 1])

    def write(self, slots, pairs, k, v):
        for src, dst in pairs:
            self.st.copy_block(src, dst)
        self.st.reshape_and_cache(0, k[0], v[0], slots)
        self.run.write(np.asarray(slots, dtype=np.int64), np.asarray(pairs, dtype=np.int32)
                       .reshape(-1, 2), k, v)

    def match(self, seq, toks):
        m = self.orc.match_prefix(seq, toks)
        assert self.c.seq_match_prefix(seq, toks) == m
        self.run.lengths[seq] = m
        return m

    def append(self, seq, toks):
        so, po = self.orc.append_tokens(seq, len(toks), toks)
        sc, pc = self.c.seq_append_tokens(seq, len(toks), toks)
        assert list(sc) == list(so) and [tuple(p) for p in pc] == list(po)
        self.run.lengths[seq] = self.run.lengths.get(seq, 0) + len(toks)
        if toks:
            k, v = self.values(len(toks))
            self.write(so, po, k, v)

    def release(self, seq):
        self.orc.release(seq)
        self.c.seq_release(seq)
        self.run.lengths.pop(seq)

    def same_pools(self):
        from paged_kv_cache_65_gb300.driver import to_host_bits

        assert np.array_equal(to_host_bits(self.c.k), self.st.K)
        assert np.array_equal(to_host_bits(self.c.v), self.st.V)
        assert self.c.kv_prefix_stats() == (self.orc.cache_stats()[3], self.orc.cache_stats()[2])
        self.c.kv_pool_check()
        self.orc.check()

    def decode(self, seqs, toks):
        """One decode step of ``seqs`` (token ids ``toks``) on both sides;
        the GPU attends per sequence and through the plan on both tensor
        passes, each compared with the oracle."""
        from paged_kv_cache_65_gb300 import _lib
        from paged_kv_cache_65_gb300.driver import to_device

        so, po = self.orc.append_slots(seqs, toks)
        sc, pc = self.c.seq_append_slots(seqs, toks)
        assert list(sc) == list(so) and [tuple(p) for p in pc] == list(po)
        for s in seqs:
            self.run.lengths[s] += 1
        k, v = self.values(len(seqs))
        self.write(so, po, k, v)
        self.calls += 1
        q = synth.storage_values(synth.normal_f32((SEED, 2, self.calls), (len(seqs), HQ, D)),
                                 "bf16")
        ref = np.stack([decode_attention(to_f64(q[i], "bf16"),
                                         *self.st.gather(0, self.orc.tables[s],
                                                         self.orc.lengths[s]))
                        for i, s in enumerate(seqs)])
        d_table, d_lens, mb = self.run.tables(seqs)
        qd = to_device(q, "bf16", "cuda")
        self.c.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, 2)
        got = [self.run.attend(0, qd, d_table, mb, d_lens, len(seqs))]
        for path in (2, 3):
            self.c.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, path)
            h_plan, d_plan, ws = self.run.plan(seqs, mb)
            got.append(self.run.attend_planned(0, qd, d_table, mb, h_plan, d_plan, ws))
        for g in got:
            err = float(np.max(np.abs(g.cpu().numpy().astype(np.float64) - ref)))
            assert err <= TOL, err
        assert self.c.kv_pool_device_status() == 0
        return so, po


def test_prefix_hits_evictions_and_decode_on_the_device():
    pp = Pair()
    rng = np.random.default_rng(SEED)
    prompt_a = [int(x) for x in rng.integers(0, 151936, 300)]

    # A: no hit; its 18 full blocks are published as they fill
    assert pp.match(0, prompt_a) == 0
    pp.append(0, prompt_a)
    pp.decode([0], [int(rng.integers(0, 151936))])
    pp.same_pools()
    pp.release(0)  # the 18 cached blocks turn dormant; the partial tail is freed
    assert pp.c.kv_prefix_stats()[1] == 18

    # B shares A's first 250 tokens: the hit is truncated to 15 whole blocks
    prompt_b = prompt_a[:250] + [int(x) for x in rng.integers(0, 151936, 50)]
    assert pp.match(1, prompt_b) == 240
    pp.append(1, prompt_b[240:])
    # C repeats A's prompt and goes on: 18 blocks (15 shared with B, 3 revived)
    prompt_c = prompt_a + [int(x) for x in rng.integers(0, 151936, 20)]
    assert pp.match(2, prompt_c) == 288
    pp.append(2, prompt_c[288:])
    pp.same_pools()
    # one step of B and C together: the plan reads their 15 common blocks once
    for _ in range(2):
        pp.decode([1, 2], [int(x) for x in rng.integers(0, 151936, 2)])
    pp.same_pools()

    # B and C leave; D's long unrelated prompt needs more blocks than are free,
    # so dormant leaves are evicted least recently used first and reused
    pp.release(1)
    pp.release(2)
    cached_before = pp.orc.cache_stats()[3]
    free_before = len(pp.orc.free)
    prompt_d = [int(x) for x in rng.integers(0, 151936, 16 * (free_before + 6) + 5)]
    assert pp.match(3, prompt_d) == 0
    pp.append(3, prompt_d)
    assert pp.orc.cache_stats()[3] < cached_before + len(prompt_d) // B  # some were evicted
    pp.same_pools()
    # D attends over blocks that held other requests' tokens before the eviction
    pp.decode([3], [int(rng.integers(0, 151936))])
    pp.same_pools()
    pp.release(3)
    # E asks for A's prompt again: the surviving chain is shorter than 288, and
    # E's tail takes blocks evicted from D's chain
    prompt_e = prompt_a + [int(x) for x in rng.integers(0, 151936, 7)]
    m = pp.match(4, prompt_e)
    assert m % B == 0 and m < 288
    pp.append(4, prompt_e[m:])
    pp.same_pools()
    for _ in range(2):
        pp.decode([4], [int(rng.integers(0, 151936))])
    pp.same_pools()
