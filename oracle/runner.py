"""Run a ``synth`` workload recipe with the oracle's own manager, store and
attention.  TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

One decode step follows "PagedAttention 的块表与碎片控制" §10 and §07:
reserve the step's slots for every listed sequence (all or nothing), copy
any shared tail that a write would touch, write each new token's K/V into
its slot, then attend over every position up to and including the new one.
"""

from __future__ import annotations

import numpy as np

from .attention import decode_attention
from .prefill import prefill_attention
from .block_manager import BlockManager
from .kv_store import INPUT_DTYPE, KVStore, to_f64


class OracleRun:
    def __init__(self, wl, with_store: bool = True):
        self.wl = wl
        self.bm = BlockManager(wl.n_blocks, wl.block_size, wl.free_order)
        self.st = (KVStore(wl.n_layers, wl.n_blocks, wl.block_size, wl.n_kv_heads,
                           wl.head_dim, wl.dtype, k_scale=getattr(wl, "k_scale", 1.0),
                           v_scale=getattr(wl, "v_scale", 1.0)) if with_store else None)
        self.build_cows = []
        for op in wl.build_ops:
            self.apply(op)

    def apply(self, op):
        kind = op[0]
        if kind == "append":
            _, seq, n, vseed = op
            slots, cows = self.bm.append_tokens(seq, n)
            self.build_cows.extend(cows)
            if self.st is not None:
                for src, dst in cows:
                    self.st.copy_block(src, dst)
                k, v = self.wl.append_values(vseed, n)
                for layer in range(self.wl.n_layers):
                    self.st.reshape_and_cache(layer, k[layer], v[layer], slots)
        elif kind == "fork":
            self.bm.fork(op[1], op[2])
        elif kind == "release":
            self.bm.release(op[1])
        else:
            raise ValueError(kind)

    def reserve_step(self):
        """Host part of a decode step: ``(slots, cow_pairs)``."""
        return self.bm.append_slots(self.wl.decode_seqs)

    def write_step(self, step: int, slots, cows):
        q, k, v = self.wl.step_values(step)
        for src, dst in cows:
            self.st.copy_block(src, dst)
        for layer in range(self.wl.n_layers):
            self.st.reshape_and_cache(layer, k[layer], v[layer], slots)
        return q

    def attend(self, layer: int, q, seq_index=None, heads=None):
        """float64 outputs ``[n_seq, H_q, D_h]`` of one layer (or of the
        listed sequence indices / heads only)."""
        wl = self.wl
        idx = range(len(wl.decode_seqs)) if seq_index is None else seq_index
        qf = to_f64(q, INPUT_DTYPE[wl.dtype])
        out = np.zeros((len(wl.decode_seqs), wl.n_q_heads, wl.head_dim))
        for i in idx:
            s = wl.decode_seqs[i]
            K, V = self.st.gather(layer, self.bm.tables[s], self.bm.lengths[s])
            if heads is None:
                out[i] = decode_attention(qf[i], K, V)
            else:
                o = decode_attention(qf[i], K, V)
                out[i, heads] = o[heads]
        return out

    def step(self, step: int):
        """A whole decode step; returns slots, cows and per-layer outputs."""
        slots, cows = self.reserve_step()
        q = self.write_step(step, slots, cows)
        outs = [self.attend(layer, q) for layer in range(self.wl.n_layers)]
        return slots, cows, q, outs

    # ------------------------------------------------------------ prefill
    def prefill_step(self, step: int = 0):
        """Host part and writes of a chunked-prefill round: each chunk's
        slots are reserved and its K/V written (the pages compute the chunk's
        keys and values fresh and store them; written first and read back
        they are the same numbers).  Returns ``(slots per chunk, copy
        pairs, q)``."""
        q, k, v = self.wl.chunk_values(step)
        all_slots, all_cows, t = [], [], 0
        for seq, c in self.wl.chunks:
            slots, cows = self.bm.append_tokens(seq, c)
            for src, dst in cows:
                self.st.copy_block(src, dst)
            for layer in range(self.wl.n_layers):
                self.st.reshape_and_cache(layer, k[layer, t:t + c], v[layer, t:t + c], slots)
            all_slots.append(slots)
            all_cows.extend(cows)
            t += c
        return all_slots, all_cows, q

    def prefill_attend(self, layer: int, q, chunk_index=None):
        """Chunked-prefill attention of the listed chunks (default: all):
        ``{chunk index: out [c, H_q, D_h]}``."""
        offs = np.cumsum([0] + [c for _, c in self.wl.chunks])
        idx = range(len(self.wl.chunks)) if chunk_index is None else chunk_index
        qf = to_f64(q, INPUT_DTYPE[self.wl.dtype])
        res = {}
        for i in idx:
            seq, c = self.wl.chunks[i]
            n = self.bm.lengths[seq]
            K, V = self.st.gather(layer, self.bm.tables[seq], n)
            res[i] = prefill_attention(qf[offs[i]:offs[i] + c], K, V)
        return res

