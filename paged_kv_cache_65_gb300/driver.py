"""Drive a pool through the C ABI from an operation script.

``DeviceRun`` replays ``("append", seq, n, value_seed)``, ``("fork", p, c)``
and ``("release", seq)`` operations against a ``PagedKVCache`` (host block
manager calls plus the slot-write and copy-on-write kernels), and runs decode
steps in the order "PagedAttention 的块表与碎片控制" §10 prescribes: reserve
the batch's slots on the host, upload metadata, copy shared tails, write the
new tokens, attend.  Values come from a caller-supplied function; nothing
here computes any part of the method.
"""

from __future__ import annotations

import numpy as np
import torch

from .cache import PagedKVCache


def to_device(x: np.ndarray, dtype: str, device) -> torch.Tensor:
    """Input elements (float32, or bfloat16 bit patterns as uint16) to a
    device tensor of the pool's input dtype (bfloat16 for FP8 pools), bit for
    bit."""
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class DeviceRun:
    def __init__(self, cache: PagedKVCache, n_q_heads: int, stream=None):
        self.c = cache
        self.n_q_heads = n_q_heads
        self.stream = stream
        self.dev = cache.k.device
        self.lengths: dict[int, int] = {}
        self.build_cows = []
        self._ws = None
        self._stage_ws = None

    # -------------------------------------------------------------- build
    def apply(self, op, values_fn) -> None:
        kind = op[0]
        c = self.c
        if kind == "append":
            _, seq, n, vseed = op
            slots, pairs = c.seq_append_tokens(seq, n)
            if len(pairs):
                self.build_cows.extend(tuple(p) for p in pairs)
                d_pairs = torch.from_numpy(np.ascontiguousarray(pairs)).to(self.dev)
                c.cow_copy(d_pairs, len(pairs), self.stream)
            if n:
                k, v = values_fn(vseed, n)  # [L, n, H_kv, D_h] stored elements
                dk = to_device(k, c.dtype, self.dev)
                dv = to_device(v, c.dtype, self.dev)
                ds = torch.from_numpy(slots).to(self.dev)
                c.reshape_and_cache(-1, dk, dv, ds, n, self.stream)
            self.lengths[seq] = self.lengths.get(seq, 0) + n
        elif kind == "fork":
            c.seq_fork(op[1], op[2])
            self.lengths[op[2]] = self.lengths[op[1]]
        elif kind == "release":
            c.seq_release(op[1])
            self.lengths.pop(op[1], None)
        else:
            raise ValueError(kind)

    # -------------------------------------------------------------- steps
    def reserve(self, seq_ids):
        slots, pairs = self.c.seq_append_slots(seq_ids)
        for s in seq_ids:
            self.lengths[s] = self.lengths.get(s, 0) + 1
        return slots, pairs

    def max_blocks(self, seq_ids) -> int:
        B = self.c.B
        return max(1, max(-(-self.lengths[s] // B) for s in seq_ids))

    def workspace(self, n_seq: int) -> torch.Tensor:
        nbytes = self.c.paged_decode_workspace_bytes(n_seq, self.n_q_heads)
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(nbytes, dtype=torch.uint8, device=self.dev)
        return self._ws

    def write(self, slots, pairs, k_new: np.ndarray, v_new: np.ndarray) -> None:
        c = self.c
        if len(pairs):
            d_pairs = torch.from_numpy(np.ascontiguousarray(pairs)).to(self.dev)
            c.cow_copy(d_pairs, len(pairs), self.stream)
        dk = to_device(k_new, c.dtype, self.dev)
        dv = to_device(v_new, c.dtype, self.dev)
        ds = torch.from_numpy(np.ascontiguousarray(slots)).to(self.dev)
        c.reshape_and_cache(-1, dk, dv, ds, len(slots), self.stream)

    def tables(self, seq_ids, max_blocks=None):
        mb = max_blocks or self.max_blocks(seq_ids)
        table, lens = self.c.seq_block_table(seq_ids, mb)
        return (torch.from_numpy(table).to(self.dev), torch.from_numpy(lens).to(self.dev), mb)

    def attend(self, layer, q_dev, d_table, max_blocks, d_lens, n_seq, out=None,
               out_dtype=torch.float32):
        c = self.c
        if out is None:
            out = torch.empty((n_seq, self.n_q_heads, c.D), dtype=out_dtype, device=self.dev)
        c.paged_decode_attention(layer, q_dev, self.n_q_heads, d_table, max_blocks, d_lens, n_seq,
                                 out, self.workspace(n_seq), 0.0, self.stream)
        return out

    def plan(self, seq_ids, max_blocks, min_shared_tokens=0):
        """Host plan of the sharing-aware pass and its device copy."""
        buf, ws_bytes = self.c.paged_decode_plan(seq_ids, self.n_q_heads, max_blocks,
                                                 min_shared_tokens)
        return buf, torch.from_numpy(buf).to(self.dev), ws_bytes

    def attend_planned(self, layer, q_dev, d_table, max_blocks, h_plan, d_plan, ws_bytes,
                       out=None, out_dtype=torch.float32):
        c = self.c
        n_seq = int(q_dev.shape[0])
        if out is None:
            out = torch.empty((n_seq, self.n_q_heads, c.D), dtype=out_dtype, device=self.dev)
        if self._ws is None or self._ws.numel() < ws_bytes:
            self._ws = torch.empty(ws_bytes, dtype=torch.uint8, device=self.dev)
        c.paged_decode_attention_planned(layer, q_dev, self.n_q_heads, d_table, max_blocks, d_plan,
                                         h_plan, out, self._ws, 0.0, self.stream)
        return out

    def step(self, seq_ids, q: np.ndarray, k_new: np.ndarray, v_new: np.ndarray, planned=False):
        """q ``[n_seq, H_q, D_h]`` (or ``[L, n_seq, H_q, D_h]``), new K/V
        ``[L, n_seq, H_kv, D_h]``.  Returns slots, pairs and float32 outputs
        ``[L, n_seq, H_q, D_h]`` on the device."""
        slots, pairs = self.reserve(seq_ids)
        self.write(slots, pairs, k_new, v_new)
        d_table, d_lens, mb = self.tables(seq_ids)
        L = self.c.L
        qd = to_device(q, self.c.dtype, self.dev)
        outs = []
        if planned:
            h_plan, d_plan, ws_bytes = self.plan(seq_ids, mb)
        for layer in range(L):
            ql = qd[layer] if qd.dim() == 4 else qd
            if planned:
                outs.append(self.attend_planned(layer, ql, d_table, mb, h_plan, d_plan, ws_bytes))
            else:
                outs.append(self.attend(layer, ql, d_table, mb, d_lens, len(seq_ids)))
        return slots, pairs, torch.stack(outs)

    def prefill_step(self, chunks, q: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
                     out_dtype=None, max_chunk=None, scheduled=False):
        """A chunked-prefill round: for each ``(seq, c)`` of ``chunks`` reserve
        ``c`` slots, copy any shared tail, write the chunk's K/V (all layers),
        then attend the chunk's queries over the sequence's context.  ``q``
        ``[n_tok, H_q, D_h]`` (chunks in order), ``k_new, v_new [L, n_tok,
        H_kv, D_h]``.  ``scheduled`` launches the work items heaviest first
        (``paged_prefill_schedule``).  Returns the outputs ``[L, n_tok, H_q,
        D_h]``."""
        import torch

        c = self.c
        seqs = [s for s, _ in chunks]
        t = 0
        for seq, n in chunks:
            if n:
                slots, pairs = c.seq_append_tokens(seq, n)
                if len(pairs):
                    d_pairs = torch.from_numpy(np.ascontiguousarray(pairs)).to(self.dev)
                    c.cow_copy(d_pairs, len(pairs), self.stream)
                dk = to_device(np.ascontiguousarray(k_new[:, t:t + n]), c.dtype, self.dev)
                dv = to_device(np.ascontiguousarray(v_new[:, t:t + n]), c.dtype, self.dev)
                c.reshape_and_cache(-1, dk, dv, torch.from_numpy(slots).to(self.dev), n,
                                    self.stream)
            self.lengths[seq] = self.lengths.get(seq, 0) + n
            t += n
        d_table, d_lens, mb = self.tables(seqs)
        starts = np.zeros(len(chunks) + 1, dtype=np.int32)
        starts[1:] = np.cumsum([n for _, n in chunks])
        d_starts = torch.from_numpy(starts).to(self.dev)
        qd = to_device(q, c.dtype, self.dev)
        dt = out_dtype or torch.float32
        mc = max_chunk if max_chunk is not None else max([n for _, n in chunks] + [0])
        if scheduled:
            sched = c.paged_prefill_schedule(starts, d_lens.cpu().numpy(), self.n_q_heads)
            d_sched = torch.from_numpy(sched).to(self.dev)
        outs = []
        staged = c.dtype == "fp8_e4m3"  # FP8 pools: through a bfloat16 copy
        if staged:
            nbytes = c.paged_prefill_staging_bytes(len(chunks), mb)
            if self._stage_ws is None or self._stage_ws.numel() < nbytes:
                self._stage_ws = torch.empty(nbytes, dtype=torch.uint8, device=self.dev)
        for layer in range(c.L):
            out = torch.zeros((int(starts[-1]), self.n_q_heads, c.D), dtype=dt, device=self.dev)
            if staged:
                c.paged_prefill_attention_staged(
                    layer, qd, self.n_q_heads, d_table, mb, d_starts, d_lens, len(chunks), out,
                    self._stage_ws, max_chunk=0 if scheduled else mc,
                    d_sched=d_sched if scheduled else None,
                    n_items=len(sched) if scheduled else 0, stream=self.stream)
            elif scheduled:
                c.paged_prefill_attention_scheduled(layer, qd, self.n_q_heads, d_table, mb,
                                                    d_starts, d_lens, len(chunks), d_sched,
                                                    len(sched), out, 0.0, self.stream)
            else:
                c.paged_prefill_attention(layer, qd, self.n_q_heads, d_table, mb, d_starts,
                                          d_lens, len(chunks), mc, out, 0.0, self.stream)
            outs.append(out)
        return torch.stack(outs)

