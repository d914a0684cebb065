"""Workload recipes (shapes, seeds, operation scripts) and value generators.

Recipes follow the decode workloads the pages measure or size:

* ``tiny``      -- 1 layer, 4 sequences of context 7, 13, 1, 16, B = 4,
                   64 blocks, H_q = 8, H_kv = 2, D_h = 64, float32; the
                   history grows token by token, round-robin over the
                   sequences, on a seeded permutation of the free list.
* ``qwen_2k``   -- one Qwen3-8B-shaped layer (H_q = 32, H_kv = 8, D_h = 128,
                   bf16, B = 16); 37 independent sequences with context
                   uniform in [2048, 2303]; 5461 blocks (12 GiB over 36
                   layers at 64 KiB per block and layer); scattered placement.
* ``shared_8k`` -- same heads; 16 sequences of 8192 + U{0..255} tokens whose
                   first 6144 tokens (384 blocks) are one shared prefix
                   (a parent is filled, forked 16 times and released).
* ``gqa70b_32k``-- a 70B-GQA-shaped layer (H_q = 64, H_kv = 8, D_h = 128,
                   bf16, B = 16): 12 parents of 32771 tokens (a tail block
                   holding 3 of 16 slots), each forked into 4 branches while
                   the parent stays alive; every decode step appends one
                   token to each of the 48 branches.
* ``pool36``    -- 36 Qwen3-8B-shaped layers; 128 sequences with lognormal
                   context (median 4096, sigma 1.0) clipped to [256, 32768];
                   the first 32 (25 %) share a 6144-token prefix; B from
                   {8, 16, 32}; the pool holds the build plus 10 % headroom.

Chunked-prefill rounds ("KV 缓存管理", chunked-prefill section; "第 8 章 推理优化"
§8.2.3: chunks of 256 to 1024 tokens, a round budget of 4096 tokens):

* ``prefill_tiny`` -- 1 layer, H_q = 8, H_kv = 2, D_h = 128, bf16, B = 16:
                   chunks of 45, 130 and 1 tokens after histories of 0, 37
                   and 200 tokens.
* ``prefill_4k``   -- one Qwen3-8B-shaped layer; 8 prompts of 8192 tokens in
                   512-token chunks, one chunk each in this round: chunks
                   1, 2, 4, 6, 8, 10, 12 and 16 (histories 0 to 7680), 4096
                   query tokens in all.

FP8 (E4M3) pools ("第 8 章 推理优化" §8.4.2's narrower KV; values are written as
bf16 rows and stored as codes of x / scale):

* ``fp8_small``   -- 1 layer, H_q = 16, H_kv = 4, D_h = 128, B = 16, 128 blocks,
                   K scale 0.5, V scale 2.0: contexts 1, 15, 16, 17, 70 and
                   333, and two sequences forked from a 150-token prefix whose
                   parent stays alive (171 and 151 tokens; the step copies the
                   shared tail for the second).
* ``qwen_2k_fp8`` -- ``qwen_2k`` with an FP8 pool (scales 1).
* ``qwen_2k_q8``  -- ``qwen_2k`` with a q8_0 pool (one fp16 scale per 32
                   values, "第 8 章 推理优化" §8.4.2 Fig. 8-23).
* ``prefill_4k_fp8`` -- ``prefill_4k`` over an FP8 pool (scales 1).
* ``shared_8k_fp8``, ``gqa70b_32k_fp8`` -- ``shared_8k`` and ``gqa70b_32k``
                   with FP8 pools (scales 1): shared prompts and narrower KV
                   together.

Context lengths named above are the lengths after the first decode step
(the step writes its token first, then attends over every position up to
and including it).

Operation scripts are lists of tuples executed in order by whoever builds
the workload::

    ("append", seq, n_tokens, value_seed)   # n slots for seq; values drawn
                                            # from value_seed
    ("fork", parent, child)
    ("release", seq)
"""

from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np


def _seed_seq(words) -> np.random.SeedSequence:
    if isinstance(words, (int, np.integer)):
        words = [int(words)]
    return np.random.SeedSequence([int(w) & 0xFFFFFFFF for w in words])


def normal_f32(seed_words, shape) -> np.ndarray:
    """float32 N(0, 1) drawn from PCG64 seeded with ``seed_words``."""
    rng = np.random.Generator(np.random.PCG64(_seed_seq(seed_words)))
    return rng.standard_normal(size=shape, dtype=np.float32)


def torch_seed(seed_words) -> int:
    """A 63-bit seed for torch generators derived from ``seed_words``."""
    state = _seed_seq(seed_words).generate_state(1, dtype=np.uint64)
    return int(state[0]) & ((1 << 63) - 1)


def storage_dtype(dtype: str):
    """Element type of the values a caller writes (FP8 pools take bf16)."""
    return {"f32": np.float32, "bf16": np.uint16, "fp8_e4m3": np.uint16, "q8_0": np.uint16}[dtype]


def storage_values(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values as stored elements: float32 as is, or bfloat16 bit
    patterns rounded to nearest even (torch's CPU conversion)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype in ("bf16", "fp8_e4m3", "q8_0"):  # code pools are written with bf16 rows
        import torch

        t = torch.from_numpy(x).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(dtype)


def permutation(seed_words, n: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(_seed_seq(seed_words)))
    return rng.permutation(n).astype(np.int32)


@dataclass
class Workload:
    name: str
    n_layers: int
    n_blocks: int
    block_size: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: str
    seed: int
    free_order: np.ndarray | None
    build_ops: list = field(default_factory=list)
    decode_seqs: list = field(default_factory=list)
    notes: str = ""
    # FP8 pools: codes of x / scale (keyword-only: positional fields keep
    # their order in subclasses)
    k_scale: float = field(default=1.0, kw_only=True)
    v_scale: float = field(default=1.0, kw_only=True)

    @property
    def elem_bytes(self) -> float:
        """Bytes of one stored K or V element (q8_0: its code and its share
        of the group's 2-byte scale, 34 / 32)."""
        return {"f32": 4, "bf16": 2, "fp8_e4m3": 1, "q8_0": 34 / 32}[self.dtype]

    # values --------------------------------------------------------------
    def append_values(self, value_seed: int, n_tokens: int):
        """K and V of one append op, stored elements
        ``[n_layers, n_tokens, H_kv, D_h]`` each."""
        x = normal_f32((self.seed, 1, value_seed),
                       (self.n_layers, n_tokens, 2, self.n_kv_heads, self.head_dim))
        x = storage_values(x, self.dtype)
        return np.ascontiguousarray(x[:, :, 0]), np.ascontiguousarray(x[:, :, 1])

    def step_values(self, step: int):
        """q ``[n_seq, H_q, D_h]`` and new K, V ``[n_layers, n_seq, H_kv, D_h]``
        for decode step ``step`` (0-based), as stored elements."""
        n = len(self.decode_seqs)
        q = normal_f32((self.seed, 2, step), (n, self.n_q_heads, self.head_dim))
        kv = normal_f32((self.seed, 3, step),
                        (self.n_layers, n, 2, self.n_kv_heads, self.head_dim))
        q = storage_values(q, self.dtype)
        kv = storage_values(kv, self.dtype)
        return q, np.ascontiguousarray(kv[:, :, 0]), np.ascontiguousarray(kv[:, :, 1])


@dataclass
class PrefillWorkload(Workload):
    """A chunked-prefill round: after the build operations, each
    ``(seq, c)`` of ``chunks`` appends a chunk of ``c`` tokens and attends
    its ``c`` queries over the sequence's whole context."""
    chunks: list = field(default_factory=list)

    def chunk_values(self, step: int):
        """q ``[n_tok, H_q, D_h]`` (the chunks in order, each chunk's tokens
        in order) and the chunks' K, V ``[n_layers, n_tok, H_kv, D_h]``, as
        stored elements."""
        n = sum(c for _, c in self.chunks)
        q = normal_f32((self.seed, 5, step), (n, self.n_q_heads, self.head_dim))
        kv = normal_f32((self.seed, 6, step),
                        (self.n_layers, n, 2, self.n_kv_heads, self.head_dim))
        q = storage_values(q, self.dtype)
        kv = storage_values(kv, self.dtype)
        return q, np.ascontiguousarray(kv[:, :, 0]), np.ascontiguousarray(kv[:, :, 1])


def _prefill(name, seed, n_q, n_kv, hist, chunk, n_blocks):
    ops = [("append", s, h, s) for s, h in enumerate(hist) if h > 0]
    chunks = [(s, c) for s, c in enumerate(chunk)]
    return PrefillWorkload(name, 1, n_blocks, 16, n_q, n_kv, 128, "bf16", seed,
                           permutation((seed, 0), n_blocks), ops, list(range(len(hist))),
                           f"chunks {list(chunk)} after histories {list(hist)}", chunks)


def _prefill_tiny(seed: int = 6) -> Workload:
    return _prefill("prefill_tiny", seed, 8, 2, [0, 37, 200], [45, 130, 1], 64)


def _prefill_4k(seed: int = 7) -> Workload:
    hist = [512 * k for k in (0, 1, 3, 5, 7, 9, 11, 15)]
    return _prefill("prefill_4k", seed, 32, 8, hist, [512] * 8, 2048)


def _prefill_4k_fp8(seed: int = 7) -> Workload:
    return dataclasses.replace(_prefill_4k(seed), name="prefill_4k_fp8", dtype="fp8_e4m3")


def _tiny(seed: int = 0) -> Workload:
    ctx = [7, 13, 1, 16]
    ops = []
    hist = [c - 1 for c in ctx]
    vs = 0
    # round-robin growth, one token at a time, as in the interleaving test
    for t in range(max(hist)):
        for s, h in enumerate(hist):
            if t < h:
                ops.append(("append", s, 1, vs))
                vs += 1
    return Workload("tiny", 1, 64, 4, 8, 2, 64, "f32", seed,
                    permutation((seed, 0), 64), ops, list(range(4)),
                    "context lengths 7, 13, 1, 16 after the step")


def _qwen_2k(seed: int = 1, dtype: str = "bf16") -> Workload:
    n_seq, n_blocks = 37, 5461
    rng = np.random.Generator(np.random.PCG64(_seed_seq((seed, 4))))
    ctx = rng.integers(2048, 2303, size=n_seq, endpoint=True)
    ops = [("append", s, int(c) - 1, s) for s, c in enumerate(ctx)]
    name = {"bf16": "qwen_2k", "fp8_e4m3": "qwen_2k_fp8", "q8_0": "qwen_2k_q8"}[dtype]
    return Workload(name, 1, n_blocks, 16, 32, 8, 128, dtype, seed,
                    permutation((seed, 0), n_blocks), ops, list(range(n_seq)),
                    "37 independent sequences, context U[2048, 2303]")


def _qwen_2k_fp8(seed: int = 1) -> Workload:
    return _qwen_2k(seed, "fp8_e4m3")


def _qwen_2k_q8(seed: int = 1) -> Workload:
    return _qwen_2k(seed, "q8_0")


def _fp8_small(seed: int = 8) -> Workload:
    ctx = [1, 15, 16, 17, 70, 333]
    ops = [("append", s, c - 1, s) for s, c in enumerate(ctx) if c > 1]
    # a 150-token prefix (a partly filled tail block) forked into two more
    # sequences while its parent stays alive: the first append of each
    # branch copies the shared tail
    parent = 100
    ops += [("append", parent, 150, 50), ("fork", parent, 6), ("fork", parent, 7),
            ("append", 6, 20, 51)]
    return Workload("fp8_small", 1, 128, 16, 16, 4, 128, "fp8_e4m3", seed,
                    permutation((seed, 0), 128), ops, list(range(8)),
                    "contexts 1, 15, 16, 17, 70, 333, 171, 151; a 150-token shared prefix",
                    k_scale=0.5, v_scale=2.0)


def _shared_8k(seed: int = 2) -> Workload:
    n_seq, n_blocks, prefix = 16, 5461, 6144
    rng = np.random.Generator(np.random.PCG64(_seed_seq((seed, 4))))
    extra = rng.integers(0, 255, size=n_seq, endpoint=True)
    parent = 1000
    ops = [("append", parent, prefix, 0)]
    for s in range(n_seq):
        ops.append(("fork", parent, s))
    ops.append(("release", parent))
    for s in range(n_seq):
        ops.append(("append", s, 8192 + int(extra[s]) - 1 - prefix, 1 + s))
    return Workload("shared_8k", 1, n_blocks, 16, 32, 8, 128, "bf16", seed,
                    permutation((seed, 0), n_blocks), ops, list(range(n_seq)),
                    "16 sequences, 6144-token shared prefix (refcount 16)")


def _gqa70b_32k(seed: int = 3, keep_parents: bool = True) -> Workload:
    n_par, n_br, ctx0, n_blocks = 12, 4, 32771, 25600
    ops, seqs = [], []
    for i in range(n_par):
        parent = 10000 + i
        ops.append(("append", parent, ctx0, i))
        for b in range(n_br):
            child = i * n_br + b
            ops.append(("fork", parent, child))
            seqs.append(child)
        if not keep_parents:
            ops.append(("release", parent))
    return Workload("gqa70b_32k", 1, n_blocks, 16, 64, 8, 128, "bf16", seed,
                    permutation((seed, 0), n_blocks), ops, seqs,
                    "12 parents x 4 branches, shared partial tail (3 of 16)")


def _shared_8k_fp8(seed: int = 2) -> Workload:
    return dataclasses.replace(_shared_8k(seed), name="shared_8k_fp8", dtype="fp8_e4m3")


def _gqa70b_32k_fp8(seed: int = 3) -> Workload:
    return dataclasses.replace(_gqa70b_32k(seed), name="gqa70b_32k_fp8", dtype="fp8_e4m3")


def _pool36(seed: int = 4, block_size: int = 16, n_steps: int = 64) -> Workload:
    n_seq, n_share, prefix = 128, 32, 6144
    rng = np.random.Generator(np.random.PCG64(_seed_seq((seed, 4))))
    ctx = np.exp(rng.normal(np.log(4096.0), 1.0, size=n_seq))
    ctx = np.clip(np.rint(ctx), 256, 32768).astype(np.int64)
    ctx[:n_share] = np.maximum(ctx[:n_share], prefix + 1)
    parent = 100000
    ops = [("append", parent, prefix, 0)]
    for s in range(n_share):
        ops.append(("fork", parent, s))
    ops.append(("release", parent))
    for s in range(n_seq):
        have = prefix if s < n_share else 0
        ops.append(("append", s, int(ctx[s]) - 1 - have, 1 + s))
    # pool: every token of every sequence counted privately, one spare block
    # per sequence and decode step, plus 10 % headroom
    tokens = int(ctx.sum()) + n_seq * (n_steps + 2 * block_size)
    n_blocks = int(1.1 * (tokens // block_size + n_seq))
    return Workload("pool36", 36, n_blocks, block_size, 32, 8, 128, "bf16", seed,
                    permutation((seed, 0), n_blocks), ops, list(range(n_seq)),
                    f"128 lognormal sequences, 25% share a 6144 prefix, B={block_size}")


WORKLOADS = {
    "tiny": _tiny,
    "qwen_2k": _qwen_2k,
    "shared_8k": _shared_8k,
    "gqa70b_32k": _gqa70b_32k,
    "shared_8k_fp8": _shared_8k_fp8,
    "gqa70b_32k_fp8": _gqa70b_32k_fp8,
    "pool36": _pool36,
    "prefill_tiny": _prefill_tiny,
    "prefill_4k": _prefill_4k,
    "prefill_4k_fp8": _prefill_4k_fp8,
    "qwen_2k_q8": _qwen_2k_q8,
    "fp8_small": _fp8_small,
    "qwen_2k_fp8": _qwen_2k_fp8,
}


def workload(name: str, **kw) -> Workload:
    return WORKLOADS[name](**kw)


def recipe_lengths(wl: Workload) -> dict:
    """Token count of every live sequence after the build operations (an
    append adds its tokens, a fork copies the parent's count, a release
    drops the sequence).  Counting only: no block arithmetic."""
    n: dict[int, int] = {}
    for op in wl.build_ops:
        if op[0] == "append":
            n[op[1]] = n.get(op[1], 0) + op[2]
        elif op[0] == "fork":
            n[op[2]] = n[op[1]]
        elif op[0] == "release":
            n.pop(op[1], None)
    return n


def restrict(wl: Workload, seqs, n_layers: int | None = None) -> Workload:
    """The same recipe cut down to the decode sequences ``seqs`` (and the
    parents they fork from), optionally with fewer layers: a bounded sample
    of a large workload for CPU timing.  The values drawn differ (the value
    arrays have another shape); lengths, sharing and placement order do not."""
    import dataclasses

    keep = set(int(s) for s in seqs)
    # parents of kept sequences are kept too (their appends build the prefix)
    for op in reversed(wl.build_ops):
        if op[0] == "fork" and op[2] in keep:
            keep.add(op[1])
    ops = [op for op in wl.build_ops
           if (op[0] == "fork" and op[2] in keep) or (op[0] != "fork" and op[1] in keep)]
    return dataclasses.replace(wl, build_ops=ops,
                               decode_seqs=[s for s in wl.decode_seqs if s in keep],
                               n_layers=wl.n_layers if n_layers is None else n_layers)
