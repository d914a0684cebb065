"""Oracle K/V pool: slot writes, block copies and contiguous gathers.
TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Layout, from "PagedAttention 的块表与碎片控制" §06::

    K_cache, V_cache : [N_layers, N_blocks, B, H_kv, D_h]
    block_table      : [N_sequences, max_blocks_per_sequence]
    context_lens     : [N_sequences]

A token at logical position ``t`` of a sequence lives in physical block
``block_table[seq, t // B]`` at slot ``t % B`` (§03, §06).  A flattened slot
number is ``p * B + o``.

Element storage: ``"f32"`` pools hold float32 values; ``"bf16"`` pools hold
the raw 16-bit patterns (uint16).  A bf16 pattern ``h`` stands for the
float32 whose bits are ``h << 16``; ``to_f64`` widens that exactly.
``"fp8_e4m3"`` pools hold E4M3 codes (uint8) of the written values divided
by the pool's K or V scale (``oracle.fp8``); the values written are bf16
patterns, and a gather returns ``code value * scale``.  ``"q8_0"`` pools
hold int8 codes (uint8 bits) of the written values and one fp16 scale per
group of 32 values of a (slot, head) row, ``Ks`` / ``Vs [N_layers,
N_blocks, B, H_kv, D_h / 32]`` (uint16 bits; ``oracle.q8``); a gather
returns ``code * scale``.
"""

from __future__ import annotations

import numpy as np

from .fp8 import e4m3_decode, e4m3_encode
from .q8 import GROUP, q8_decode, q8_encode

STORAGE = {"f32": np.float32, "bf16": np.uint16, "fp8_e4m3": np.uint8, "q8_0": np.uint8}
# dtype of the rows a caller writes (and of q) for each pool dtype
INPUT_DTYPE = {"f32": "f32", "bf16": "bf16", "fp8_e4m3": "bf16", "q8_0": "bf16"}


def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of stored elements to float64."""
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


class KVStore:
    def __init__(self, n_layers, n_blocks, block_size, n_kv_heads, head_dim, dtype="f32",
                 k_scale=1.0, v_scale=1.0):
        self.L, self.N, self.B = n_layers, n_blocks, block_size
        self.H, self.D, self.dtype = n_kv_heads, head_dim, dtype
        self.k_scale, self.v_scale = float(k_scale), float(v_scale)
        shape = (n_layers, n_blocks, block_size, n_kv_heads, head_dim)
        self.K = np.zeros(shape, dtype=STORAGE[dtype])
        self.V = np.zeros(shape, dtype=STORAGE[dtype])
        if dtype == "q8_0":
            sshape = shape[:-1] + (head_dim // GROUP,)
            self.Ks = np.zeros(sshape, dtype=np.uint16)
            self.Vs = np.zeros(sshape, dtype=np.uint16)

    def write_slot(self, layer: int, slot: int, k_row, v_row) -> None:
        p, o = divmod(int(slot), self.B)
        if self.dtype == "q8_0":
            # rows arrive as bf16 patterns; each head's row in groups of 32
            kc, ks = q8_encode(to_f64(k_row, "bf16").astype(np.float32))
            vc, vs = q8_encode(to_f64(v_row, "bf16").astype(np.float32))
            self.K[layer, p, o], self.Ks[layer, p, o] = kc, ks
            self.V[layer, p, o], self.Vs[layer, p, o] = vc, vs
            return
        if self.dtype == "fp8_e4m3":
            # rows arrive as bf16 patterns; stored as codes of x / scale
            self.K[layer, p, o] = e4m3_encode(to_f64(k_row, "bf16").astype(np.float32), self.k_scale)
            self.V[layer, p, o] = e4m3_encode(to_f64(v_row, "bf16").astype(np.float32), self.v_scale)
            return
        self.K[layer, p, o] = k_row
        self.V[layer, p, o] = v_row

    def reshape_and_cache(self, layer: int, k_new, v_new, slots) -> None:
        """Token ``i``'s rows ``[H_kv, D_h]`` go to slot ``slots[i]``; a
        negative slot means "no write" for that token."""
        for i, s in enumerate(slots):
            if s < 0:
                continue
            self.write_slot(layer, s, k_new[i], v_new[i])

    def copy_block(self, src: int, dst: int) -> None:
        """Copy-on-write copy: every slot of block ``src`` in every layer,
        K and V, into block ``dst``."""
        self.K[:, dst] = self.K[:, src]
        self.V[:, dst] = self.V[:, src]
        if self.dtype == "q8_0":
            self.Ks[:, dst] = self.Ks[:, src]
            self.Vs[:, dst] = self.Vs[:, src]

    def gather_raw(self, layer: int, table, ctx: int):
        """Positions ``0..ctx-1`` of one sequence, in logical order, as
        stored elements ``[ctx, H_kv, D_h]``.  Taken block by block: logical
        block ``j`` holds positions ``j*B .. j*B + B - 1`` in slots ``0..B-1``
        of physical block ``table[j]``, the last one only its first
        ``ctx - j*B`` slots."""
        ks, vs = [], []
        for j in range(-(-ctx // self.B)):
            p = table[j]
            rows = min(self.B, ctx - j * self.B)
            ks.append(self.K[layer, p, :rows])
            vs.append(self.V[layer, p, :rows])
        shape = (0, self.H, self.D)
        k = np.concatenate(ks) if ks else np.zeros(shape, dtype=self.K.dtype)
        v = np.concatenate(vs) if vs else np.zeros(shape, dtype=self.V.dtype)
        return k, v

    def gather(self, layer: int, table, ctx: int):
        """Same as ``gather_raw`` but widened to contiguous float64 (FP8
        codes dequantized: value times the pool's scale, exact)."""
        k, v = self.gather_raw(layer, table, ctx)
        if self.dtype == "fp8_e4m3":
            return e4m3_decode(k) * self.k_scale, e4m3_decode(v) * self.v_scale
        if self.dtype == "q8_0":
            ks, vs = [], []
            for j in range(-(-ctx // self.B)):
                rows = min(self.B, ctx - j * self.B)
                ks.append(self.Ks[layer, table[j], :rows])
                vs.append(self.Vs[layer, table[j], :rows])
            shape = (0, self.H, self.D // GROUP)
            sk = np.concatenate(ks) if ks else np.zeros(shape, dtype=np.uint16)
            sv = np.concatenate(vs) if vs else np.zeros(shape, dtype=np.uint16)
            return q8_decode(k, sk), q8_decode(v, sv)
        return to_f64(k, self.dtype), to_f64(v, self.dtype)
