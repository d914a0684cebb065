"""Python face of the C ABI: one object per pool.

``PagedKVCache`` owns the device tensors (allocated with torch: K and V pools
``[N_layers, N_blocks, B, H_kv, D_h]`` and a status word) and the library's
pool handle.  Each method forwards to the C function of the same name;
nothing here computes any part of the method.
"""

from __future__ import annotations

import ctypes as C

import numpy as np

from . import _lib
from ._lib import check, i32, lib, ptr_f32, ptr_i32, ptr_i64, vp

DTYPES = {"f32": _lib.KV_DTYPE_F32, "bf16": _lib.KV_DTYPE_BF16, "fp8_e4m3": _lib.KV_DTYPE_FP8_E4M3,
          "q8_0": _lib.KV_DTYPE_Q8_0}


def _stream(stream) -> C.c_void_p:
    if stream is None:
        try:
            import torch

            if torch.cuda.is_available():
                return C.c_void_p(torch.cuda.current_stream().cuda_stream)
        except Exception:  # pragma: no cover - torch always present here
            pass
        return C.c_void_p(0)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


class PagedKVCache:
    def __init__(self, n_layers, n_blocks, block_size, n_kv_heads, head_dim, dtype="bf16",
                 device="cuda", free_order=None, allocate=True, k_cache=None, v_cache=None):
        self.L, self.N, self.B = n_layers, n_blocks, block_size
        self.H, self.D, self.dtype = n_kv_heads, head_dim, dtype
        self.k = k_cache
        self.v = v_cache
        self.k_sc = self.v_sc = None  # q8_0: fp16 scales [L, N, H_kv, B, D_h / 32]
        self.status = None
        if allocate and k_cache is None:
            import torch

            tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8_e4m3": torch.uint8,
                   "q8_0": torch.uint8}[dtype]
            shape = (n_layers, n_blocks, block_size, n_kv_heads, head_dim)
            self.k = torch.empty(shape, dtype=tdt, device=device)
            self.v = torch.empty(shape, dtype=tdt, device=device)
            if dtype == "q8_0":
                sshape = (n_layers, n_blocks, n_kv_heads, block_size, head_dim // 32)
                self.k_sc = torch.zeros(sshape, dtype=torch.float16, device=device)
                self.v_sc = torch.zeros(sshape, dtype=torch.float16, device=device)
        if self.k is not None:
            import torch

            self.status = torch.zeros(1, dtype=torch.int32, device=self.k.device)
        order = None if free_order is None else i32(free_order)
        h = C.c_void_p()
        check(lib.kv_pool_create(n_layers, n_blocks, block_size, n_kv_heads, head_dim,
                                 DTYPES[dtype], vp(self.k), vp(self.v), vp(self.status),
                                 ptr_i32(order) if order is not None else None, C.byref(h)),
              "kv_pool_create")
        self.handle = h
        if self.k_sc is not None:
            check(lib.kv_pool_set_q8_scales(h, vp(self.k_sc), vp(self.v_sc)),
                  "kv_pool_set_q8_scales")

    def close(self):
        if getattr(self, "handle", None):
            lib.kv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ host
    def kv_pool_stats(self):
        f, a, s = C.c_int(), C.c_int(), C.c_int()
        check(lib.kv_pool_stats(self.handle, C.byref(f), C.byref(a), C.byref(s)), "kv_pool_stats")
        return f.value, a.value, s.value

    def kv_pool_check(self):
        check(lib.kv_pool_check(self.handle), "kv_pool_check")

    def kv_pool_set_option(self, option, value):
        check(lib.kv_pool_set_option(self.handle, int(option), int(value)), "kv_pool_set_option")

    def kv_pool_set_fp8_scales(self, k_scale, v_scale):
        check(lib.kv_pool_set_fp8_scales(self.handle, float(k_scale), float(v_scale)),
              "kv_pool_set_fp8_scales")

    def kv_block_refcount(self, block_id):
        out = C.c_int()
        check(lib.kv_block_refcount(self.handle, int(block_id), C.byref(out)), "kv_block_refcount")
        return out.value

    def block_alloc(self, n):
        out = np.zeros(max(n, 1), dtype=np.int32)
        check(lib.block_alloc(self.handle, n, ptr_i32(out)), "block_alloc")
        return out[:n]

    def block_free(self, ids):
        a = i32(ids)
        check(lib.block_free(self.handle, ptr_i32(a), a.size), "block_free")

    def block_fork(self, ids):
        a = i32(ids)
        check(lib.block_fork(self.handle, ptr_i32(a), a.size), "block_fork")

    def block_cow(self, block_id):
        out = C.c_int32()
        check(lib.block_cow(self.handle, int(block_id), C.byref(out)), "block_cow")
        return out.value

    def seq_append_slots(self, seq_ids, token_ids=None):
        """One slot per listed sequence; ``token_ids`` (one per sequence) feed
        the prefix cache."""
        ids = i32(seq_ids)
        n = ids.size
        slots = np.zeros(max(n, 1), dtype=np.int64)
        pairs = np.zeros((max(n, 1), 2), dtype=np.int32)
        ncow = C.c_int()
        if token_ids is None:
            check(lib.seq_append_slots(self.handle, ptr_i32(ids), n, ptr_i64(slots),
                                       ptr_i32(pairs), C.byref(ncow)), "seq_append_slots")
        else:
            toks = i32(token_ids)
            if toks.size != n:
                raise ValueError("token_ids: one per sequence")
            check(lib.seq_append_slots_ids(self.handle, ptr_i32(ids), n, ptr_i32(toks),
                                           ptr_i64(slots), ptr_i32(pairs), C.byref(ncow)),
                  "seq_append_slots_ids")
        return slots[:n], pairs[:ncow.value]

    def seq_append_tokens(self, seq, n_tokens, token_ids=None):
        slots = np.zeros(max(n_tokens, 1), dtype=np.int64)
        pair = np.zeros(2, dtype=np.int32)
        ncow = C.c_int()
        if token_ids is None:
            check(lib.seq_append_tokens(self.handle, int(seq), int(n_tokens), ptr_i64(slots),
                                        ptr_i32(pair), C.byref(ncow)), "seq_append_tokens")
        else:
            toks = i32(token_ids)
            if toks.size != n_tokens:
                raise ValueError("token_ids: one per token")
            check(lib.seq_append_tokens_ids(self.handle, int(seq), int(n_tokens),
                                            ptr_i32(np.ascontiguousarray(toks)) if n_tokens else
                                            ptr_i32(np.zeros(1, dtype=np.int32)),
                                            ptr_i64(slots), ptr_i32(pair), C.byref(ncow)),
                  "seq_append_tokens_ids")
        return slots[:n_tokens], pair.reshape(1, 2)[:ncow.value]

    # ------------------------------------------------------ prefix cache
    def kv_prefix_cache_enable(self, salt=0):
        check(lib.kv_prefix_cache_enable(self.handle, int(salt) & ((1 << 64) - 1)),
              "kv_prefix_cache_enable")

    def seq_match_prefix(self, seq, tokens):
        toks = i32(tokens)
        out = C.c_int()
        buf = toks if toks.size else np.zeros(1, dtype=np.int32)
        check(lib.seq_match_prefix(self.handle, int(seq), ptr_i32(buf), int(toks.size),
                                   C.byref(out)), "seq_match_prefix")
        return out.value

    def kv_prefix_evict(self, target_free):
        out = C.c_int()
        check(lib.kv_prefix_evict(self.handle, int(target_free), C.byref(out)), "kv_prefix_evict")
        return out.value

    def kv_prefix_stats(self):
        cached, dormant = C.c_int(), C.c_int()
        check(lib.kv_prefix_stats(self.handle, C.byref(cached), C.byref(dormant)),
              "kv_prefix_stats")
        return cached.value, dormant.value

    def seq_fork(self, parent, child):
        check(lib.seq_fork(self.handle, int(parent), int(child)), "seq_fork")

    def seq_release(self, seq):
        check(lib.seq_release(self.handle, int(seq)), "seq_release")

    def seq_length(self, seq):
        out = C.c_int()
        check(lib.seq_length(self.handle, int(seq), C.byref(out)), "seq_length")
        return out.value

    def seq_block_table(self, seq_ids, max_blocks):
        ids = i32(seq_ids)
        n = ids.size
        table = np.zeros((max(n, 1), max(max_blocks, 1)), dtype=np.int32)
        lens = np.zeros(max(n, 1), dtype=np.int32)
        check(lib.seq_block_table(self.handle, ptr_i32(ids), n, max_blocks, ptr_i32(table),
                                  ptr_i32(lens)), "seq_block_table")
        return table[:n, :max_blocks], lens[:n]

    # ---------------------------------------------------------- device
    def kv_pool_device_status(self, stream=None):
        bits = C.c_int()
        st = lib.kv_pool_device_status(self.handle, _stream(stream), C.byref(bits))
        if st not in (_lib.KV_OK, _lib.KV_ERR_DEVICE_CHECK):
            check(st, "kv_pool_device_status")
        return bits.value

    def kv_device_wait_selftest(self, limit_us, stream=None):
        check(lib.kv_device_wait_selftest(self.handle, int(limit_us), _stream(stream)),
              "kv_device_wait_selftest")

    def cow_copy(self, d_pairs, n_pairs, stream=None):
        check(lib.cow_copy(self.handle, vp(d_pairs), int(n_pairs), _stream(stream)), "cow_copy")

    def reshape_and_cache(self, layer, k_new, v_new, d_slots, n_tokens, stream=None):
        check(lib.reshape_and_cache(self.handle, int(layer), vp(k_new), vp(v_new), vp(d_slots),
                                    int(n_tokens), _stream(stream)), "reshape_and_cache")

    def paged_decode_workspace_bytes(self, n_seq, n_q_heads):
        return int(lib.paged_decode_workspace_bytes(self.handle, int(n_seq), int(n_q_heads)))

    def paged_decode_partials(self, layer, q, n_q_heads, d_table, max_blocks, d_lens, n_seq,
                              workspace, scale=0.0, stream=None):
        check(lib.paged_decode_partials(self.handle, int(layer), vp(q), int(n_q_heads), vp(d_table),
                                        int(max_blocks), vp(d_lens), int(n_seq), float(scale),
                                        vp(workspace), _nbytes(workspace), _stream(stream)),
              "paged_decode_partials")

    def paged_decode_merge(self, n_q_heads, d_lens, n_seq, out, workspace, stream=None):
        check(lib.paged_decode_merge(self.handle, int(n_q_heads), vp(d_lens), int(n_seq), vp(out),
                                     _out_dtype(out), vp(workspace), _nbytes(workspace),
                                     _stream(stream)), "paged_decode_merge")

    def paged_decode_attention(self, layer, q, n_q_heads, d_table, max_blocks, d_lens, n_seq, out,
                               workspace, scale=0.0, stream=None):
        check(lib.paged_decode_attention(self.handle, int(layer), vp(q), int(n_q_heads),
                                         vp(d_table), int(max_blocks), vp(d_lens), int(n_seq),
                                         float(scale), vp(out), _out_dtype(out), vp(workspace),
                                         _nbytes(workspace), _stream(stream)),
              "paged_decode_attention")

    def paged_decode_plan(self, seq_ids, n_q_heads, max_blocks, min_shared_tokens=0):
        """Host plan of a sharing-aware decode pass: (plan bytes, workspace bytes)."""
        ids = i32(seq_ids)
        cap = int(lib.paged_decode_plan_bytes(self.handle, ids.size, int(n_q_heads)))
        buf = np.zeros(max(cap, 16), dtype=np.uint8)
        ws = C.c_size_t()
        check(lib.paged_decode_plan(self.handle, ptr_i32(ids), ids.size, int(n_q_heads),
                                    int(max_blocks), int(min_shared_tokens), vp(buf), buf.nbytes,
                                    C.byref(ws)), "paged_decode_plan")
        return buf, int(ws.value)

    def paged_decode_partials_planned(self, layer, q, n_q_heads, d_table, max_blocks, d_plan,
                                      h_plan, workspace, scale=0.0, stream=None):
        check(lib.paged_decode_partials_planned(self.handle, int(layer), vp(q), int(n_q_heads),
                                                vp(d_table), int(max_blocks), vp(d_plan),
                                                vp(h_plan), float(scale), vp(workspace),
                                                _nbytes(workspace), _stream(stream)),
              "paged_decode_partials_planned")

    def paged_decode_partials_planned_write(self, layer, q, n_q_heads, k_new, v_new, d_table,
                                            max_blocks, d_plan, h_plan, workspace, scale=0.0,
                                            stream=None):
        """The planned split pass with this layer's slot write of the step's
        newest tokens (rows of ``k_new``, ``v_new`` in plan order) fused in."""
        check(lib.paged_decode_partials_planned_write(
            self.handle, int(layer), vp(q), int(n_q_heads), vp(k_new), vp(v_new), vp(d_table),
            int(max_blocks), vp(d_plan), vp(h_plan), float(scale), vp(workspace),
            _nbytes(workspace), _stream(stream)), "paged_decode_partials_planned_write")

    def paged_decode_merge_planned(self, n_q_heads, d_plan, h_plan, out, workspace, stream=None):
        check(lib.paged_decode_merge_planned(self.handle, int(n_q_heads), vp(d_plan), vp(h_plan),
                                             vp(out), _out_dtype(out), vp(workspace),
                                             _nbytes(workspace), _stream(stream)),
              "paged_decode_merge_planned")

    def paged_decode_attention_planned(self, layer, q, n_q_heads, d_table, max_blocks, d_plan,
                                       h_plan, out, workspace, scale=0.0, stream=None):
        check(lib.paged_decode_attention_planned(self.handle, int(layer), vp(q), int(n_q_heads),
                                                 vp(d_table), int(max_blocks), vp(d_plan),
                                                 vp(h_plan), float(scale), vp(out),
                                                 _out_dtype(out), vp(workspace),
                                                 _nbytes(workspace), _stream(stream)),
              "paged_decode_attention_planned")

    def paged_decode_attention_noalloc(self, layer, q, n_q_heads, d_table, max_blocks, d_lens,
                                       n_seq, out, scale=0.0, stream=None):
        """Decode attention with the library's static scratch instead of a
        caller workspace (for callers that cannot allocate device memory)."""
        check(lib.paged_decode_attention_noalloc(self.handle, int(layer), vp(q), int(n_q_heads),
                                                 vp(d_table), int(max_blocks), vp(d_lens),
                                                 int(n_seq), float(scale), vp(out),
                                                 _out_dtype(out), _stream(stream)),
              "paged_decode_attention_noalloc")

    def paged_prefill_attention(self, layer, q, n_q_heads, d_table, max_blocks, d_chunk_start,
                                d_context_lens, n_seq, max_chunk, out, scale=0.0, stream=None):
        """Chunked-prefill attention of each sequence's chunk (rows
        ``d_chunk_start[s] .. d_chunk_start[s + 1] - 1`` of ``q``) over its
        paged context; the chunks' K/V must already be in the pool."""
        check(lib.paged_prefill_attention(self.handle, int(layer), vp(q), int(n_q_heads),
                                          vp(d_table), int(max_blocks), vp(d_chunk_start),
                                          vp(d_context_lens), int(n_seq), int(max_chunk),
                                          float(scale), vp(out), _out_dtype(out),
                                          _stream(stream)),
              "paged_prefill_attention")

    def paged_prefill_schedule(self, chunk_start, context_lens, n_q_heads):
        """Heaviest-first order of the prefill work items from host copies of
        the chunk geometry: int32 ``[n_items, 4]`` records (sequence, tile,
        chunk length, 128-key blocks)."""
        st = i32(chunk_start)
        ctx = i32(context_lens)
        n_seq = ctx.size
        if st.size != n_seq + 1:
            raise ValueError("chunk_start needs n_seq + 1 entries")
        mc = int(np.max(np.diff(st))) if n_seq else 0
        cap = int(lib.paged_prefill_schedule_bytes(self.handle, n_seq, int(n_q_heads), max(mc, 0)))
        buf = np.zeros((max(cap, 16) + 15) // 16 * 4, dtype=np.int32)
        n = C.c_int()
        check(lib.paged_prefill_schedule(self.handle, ptr_i32(st), ptr_i32(ctx), n_seq,
                                         int(n_q_heads), vp(buf), buf.nbytes, C.byref(n)),
              "paged_prefill_schedule")
        return buf[: 4 * n.value].reshape(n.value, 4).copy()

    def paged_prefill_schedule_bytes_for(self, chunk_start, n_q_heads):
        """Bytes of a work order for this chunk geometry's longest chunk."""
        st = i32(chunk_start)
        mc = int(np.max(np.diff(st))) if st.size > 1 else 0
        return int(lib.paged_prefill_schedule_bytes(self.handle, st.size - 1, int(n_q_heads), mc))

    def paged_prefill_attention_scheduled(self, layer, q, n_q_heads, d_table, max_blocks,
                                          d_chunk_start, d_context_lens, n_seq, d_sched, n_items,
                                          out, scale=0.0, stream=None):
        """paged_prefill_attention over a heaviest-first work order (the
        device copy of ``paged_prefill_schedule``'s records)."""
        check(lib.paged_prefill_attention_scheduled(self.handle, int(layer), vp(q),
                                                    int(n_q_heads), vp(d_table), int(max_blocks),
                                                    vp(d_chunk_start), vp(d_context_lens),
                                                    int(n_seq), vp(d_sched), int(n_items),
                                                    float(scale), vp(out), _out_dtype(out),
                                                    _stream(stream)),
              "paged_prefill_attention_scheduled")

    def paged_prefill_staging_bytes(self, n_seq, max_blocks):
        return int(lib.paged_prefill_staging_bytes(self.handle, int(n_seq), int(max_blocks)))

    def paged_prefill_attention_staged(self, layer, q, n_q_heads, d_table, max_blocks,
                                       d_chunk_start, d_context_lens, n_seq, out, workspace,
                                       max_chunk=0, d_sched=None, n_items=0, scale=0.0,
                                       stream=None):
        """Chunked prefill for any pool dtype (an FP8 pool through a bfloat16
        copy in ``workspace``); natural grid over ``max_chunk``, or the work
        order ``d_sched`` of ``n_items`` records."""
        check(lib.paged_prefill_attention_staged(
            self.handle, int(layer), vp(q), int(n_q_heads), vp(d_table), int(max_blocks),
            vp(d_chunk_start), vp(d_context_lens), int(n_seq), int(max_chunk), vp(d_sched),
            int(n_items), float(scale), vp(out), _out_dtype(out), vp(workspace),
            _nbytes(workspace) if workspace is not None else 0, _stream(stream)),
            "paged_prefill_attention_staged")

    def kv_decode_step_staging_bytes(self, n_seq, n_q_heads, max_blocks):
        return int(lib.kv_decode_step_staging_bytes(self.handle, int(n_seq), int(n_q_heads),
                                                    int(max_blocks)))

    def kv_decode_step_host(self, seq_ids, n_q_heads, max_blocks, h_q, h_k_new, h_v_new, h_out,
                            staging, scale=0.0, stream=None):
        ids = seq_ids
        if ids is self._step_ids:
            addr = self._step_ids_addr  # the same int32 array as last call: same buffer
        else:
            if not (isinstance(ids, np.ndarray) and ids.dtype == np.int32
                    and ids.flags.c_contiguous):
                ids = i32(seq_ids)
            addr = ids.ctypes.data
            if ids is seq_ids:  # the caller's own array: kept, so its buffer stays put
                self._step_ids, self._step_ids_addr = ids, addr
        check(lib.kv_decode_step_host(self.handle, addr, ids.size, n_q_heads,
                                      max_blocks, _addr(h_q), _addr(h_k_new), _addr(h_v_new),
                                      scale, _addr(h_out), _addr(staging), _nbytes(staging),
                                      self._raw_stream() if stream is None else _stream(stream)),
              "kv_decode_step_host")

    _step_ids = None
    _step_ids_addr = 0
    _stream_fn = None

    def _raw_stream(self) -> int:
        """The current torch stream of this pool's device as a raw handle."""
        if self._stream_fn is None:
            import torch

            dev = self.k.device.index if self.k is not None and self.k.device.index is not None \
                else torch.cuda.current_device()
            raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
            self._stream_fn = (lambda: raw(dev)) if raw is not None else \
                (lambda: torch.cuda.current_stream(dev).cuda_stream)
        return self._stream_fn()


def _addr(x) -> int:
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return x.ctypes.data


def _nbytes(t) -> int:
    if hasattr(t, "numel"):
        return t.numel() * t.element_size()
    return t.nbytes


def _out_dtype(out) -> int:
    import torch

    if out.dtype == torch.float32:
        return _lib.KV_DTYPE_F32
    if out.dtype == torch.bfloat16:
        return _lib.KV_DTYPE_BF16
    raise TypeError(out.dtype)


PLAN_SEG = np.dtype([("wpre", "<i8"), ("rep", "<i4"), ("b0", "<i4"), ("b1", "<i4"),
                     ("tok_end", "<i4"), ("head", "<i4"), ("ncols", "<i4"), ("mem", "<i4"),
                     ("w", "<i4")])
PLAN_ENTRY = np.dtype([("seg", "<i4"), ("col_base", "<i4")])
PLAN_START = np.dtype([("seg", "<i4"), ("rep", "<i4"), ("head", "<i4"), ("b0", "<i4"),
                       ("b1", "<i4"), ("tok_end", "<i4"), ("ncols", "<i4"), ("mem", "<i4"),
                       ("r_after", "<i8"), ("n_pid", "<i4"), ("last", "<i4"),
                       ("pid", "<i4", (16,)), ("pad1", "<i4", (4,))])


def parse_plan(buf: np.ndarray) -> dict:
    """Read a plan built by ``paged_decode_plan`` (layout of csrc/plan.h)."""
    h = np.frombuffer(buf[:80].tobytes(), dtype=np.int32)
    W = int(np.frombuffer(buf[:8].tobytes(), dtype=np.int64)[0])
    (n_segs, n_members, n_entries, c_max, n_seq, n_kv_heads, group, block_size, seg_off,
     mem_off, eoff_off, ent_off, n_shared, kernel, start_off, start_grid) = (
        int(x) for x in h[2:18])
    segs = np.frombuffer(buf[seg_off:seg_off + 40 * n_segs].tobytes(), dtype=PLAN_SEG)
    members = np.frombuffer(buf[mem_off:mem_off + 4 * n_members].tobytes(), dtype=np.int32)
    eoff = np.frombuffer(buf[eoff_off:eoff_off + 4 * (n_seq * n_kv_heads + 1)].tobytes(),
                         dtype=np.int32)
    ents = np.frombuffer(buf[ent_off:ent_off + 8 * n_entries].tobytes(), dtype=PLAN_ENTRY)
    starts = np.frombuffer(buf[start_off:start_off + 128 * start_grid].tobytes(),
                           dtype=PLAN_START)
    return dict(W=W, n_segs=n_segs, c_max=c_max, n_seq=n_seq, H=n_kv_heads, G=group,
                B=block_size, n_shared_segs=n_shared, kernel=kernel, segs=segs,
                members=members, eoff=eoff, ents=ents, start_grid=start_grid, starts=starts)
