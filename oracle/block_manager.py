"""Oracle block manager: FIFO free list, block tables, reference counts,
fork and copy-on-write.  TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources, by page title and section:

* "PagedAttention 的块表与碎片控制" §03 -- address translation
  ``j = t // B``, ``r = t % B``, ``p = block_table[j]``.
* same page §04 -- a new physical block is taken from the free list only when
  the tail block is full (``offset == 0``); so at most ``B - 1`` slots of the
  last block are ever unused.
* same page §05 -- the teaching ``BlockManager``: ``free`` is a deque of
  block ids ``0..N-1``, allocation is ``popleft`` and release is ``append``
  (FIFO); ``append_slot`` returns ``(physical_block, offset)`` and raises when
  the free list is empty.
* same page §08 and "KV 缓存管理", section "通过写时复制分支实现零复制审慎推理"
  -- per-block reference counts; ``fork`` copies the parent's table, adds one
  reference to every block in it and registers the child with the parent's
  length; a write into a tail block whose count is above one first takes a
  fresh block, copies the shared block into it, drops one reference from the
  shared block and remaps the table entry; ``release`` walks the table in
  order, drops one reference per entry and returns blocks that reach zero to
  the free list.
* "PagedAttention 的块表与碎片控制" §10 -- the new blocks a step needs are
  reserved atomically before any kernel runs: a batch either succeeds whole
  or changes nothing.
* same page §13 -- the conservation checks ``N_free + N_allocated = N_total``
  and "the set of blocks with a positive count is exactly the allocated set".

Readings where the pages leave a step open:

* A batch is processed in the order the caller lists its sequences; the first
  of several sharers of a partially filled tail to write copies, and once the
  count drops to one the last sharer writes in place.
* The copy-on-write copies the whole block (all ``B`` slots, K and V, every
  layer); only the filled slots matter.
* Block-level handles (``alloc``/``free``/``incref``/``cow``) are references
  held by the caller rather than by a table.  ``ref[p]`` is always the number
  of table entries naming ``p`` plus the caller-held handles on ``p``.
* Releasing or forking from an unknown sequence, forking onto an existing
  one, or listing a sequence twice in one batch is an invalid argument.
"""

from __future__ import annotations

import copy
from collections import deque


class NoFreeBlock(MemoryError):
    """The free list is empty (the teaching manager's ``MemoryError``)."""


class InvalidArg(ValueError):
    pass


class RefcountError(RuntimeError):
    pass


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise InvalidArg("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        if free_order is None:
            free_order = range(num_blocks)
        free_order = [int(p) for p in free_order]
        if sorted(free_order) != list(range(num_blocks)):
            raise InvalidArg("free_order must be a permutation of 0..N-1")
        self.free = deque(free_order)
        self.ref = [0] * num_blocks
        self.ext = [0] * num_blocks  # references held by block-level callers
        self.tables: dict[int, list[int]] = {}
        self.lengths: dict[int, int] = {}

    # ------------------------------------------------------------------
    # sequence level
    # ------------------------------------------------------------------
    def _pop_free(self) -> int:
        if not self.free:
            raise NoFreeBlock("no free KV block")
        return self.free.popleft()

    def append_slot(self, seq: int):
        """One token for ``seq``.  Returns ``(p, o, cow)`` where ``cow`` is
        ``(src, dst)`` when a shared tail had to be copied, else ``None``."""
        table = self.tables.setdefault(seq, [])
        length = self.lengths.get(seq, 0)
        j, r = divmod(length, self.block_size)
        cow = None
        if j == len(table):
            p = self._pop_free()
            self.ref[p] = 1
            table.append(p)
        elif self.ref[table[j]] > 1:
            old = table[j]
            new = self._pop_free()
            self.ref[old] -= 1
            self.ref[new] = 1
            table[j] = new
            cow = (old, new)
        self.lengths[seq] = length + 1
        return table[j], r, cow

    def _snapshot(self):
        return copy.deepcopy((self.free, self.ref, self.ext, self.tables, self.lengths))

    def _restore(self, snap):
        self.free, self.ref, self.ext, self.tables, self.lengths = snap

    def append_slots(self, seq_ids):
        """One token for each listed sequence, all or nothing.
        Returns ``(slots, cow_pairs)`` with ``slot = p * B + o``."""
        seq_ids = [int(s) for s in seq_ids]
        if len(set(seq_ids)) != len(seq_ids):
            raise InvalidArg("a sequence is listed twice in one batch")
        snap = self._snapshot()
        slots, cows = [], []
        try:
            for s in seq_ids:
                p, o, cow = self.append_slot(s)
                slots.append(p * self.block_size + o)
                if cow is not None:
                    cows.append(cow)
        except NoFreeBlock:
            self._restore(snap)
            raise
        return slots, cows

    def append_tokens(self, seq: int, n: int):
        """``n`` tokens for one sequence (a prefill chunk), all or nothing."""
        if n < 0:
            raise InvalidArg("negative token count")
        snap = self._snapshot()
        slots, cows = [], []
        try:
            for _ in range(n):
                p, o, cow = self.append_slot(seq)
                slots.append(p * self.block_size + o)
                if cow is not None:
                    cows.append(cow)
        except NoFreeBlock:
            self._restore(snap)
            raise
        return slots, cows

    def fork(self, parent: int, child: int) -> None:
        if parent not in self.lengths:
            raise InvalidArg("unknown parent sequence")
        if child in self.lengths or child in self.tables:
            raise InvalidArg("child sequence already exists")
        self.tables[child] = list(self.tables.get(parent, []))
        for p in self.tables[child]:
            self.ref[p] += 1
        self.lengths[child] = self.lengths[parent]

    def release(self, seq: int) -> None:
        if seq not in self.lengths:
            raise InvalidArg("unknown sequence")
        for p in self.tables.pop(seq, []):
            self.ref[p] -= 1
            if self.ref[p] == 0:
                self.free.append(p)
        self.lengths.pop(seq)

    # ------------------------------------------------------------------
    # block level (caller-held handles)
    # ------------------------------------------------------------------
    def alloc(self, n: int):
        if n < 0:
            raise InvalidArg("negative count")
        if n > len(self.free):
            raise NoFreeBlock("no free KV block")
        out = []
        for _ in range(n):
            p = self.free.popleft()
            self.ref[p] = 1
            self.ext[p] = 1
            out.append(p)
        return out

    def _check_ids(self, ids):
        for p in ids:
            if not 0 <= p < self.num_blocks:
                raise InvalidArg("block id out of range")

    def free_blocks(self, ids) -> None:
        ids = [int(p) for p in ids]
        self._check_ids(ids)
        need: dict[int, int] = {}
        for p in ids:
            need[p] = need.get(p, 0) + 1
        for p, k in need.items():
            if self.ext[p] < k:
                raise RefcountError("releasing a handle that is not held")
        for p in ids:
            self.ref[p] -= 1
            self.ext[p] -= 1
            if self.ref[p] == 0:
                self.free.append(p)

    def incref(self, ids) -> None:
        ids = [int(p) for p in ids]
        self._check_ids(ids)
        for p in ids:
            if self.ref[p] == 0:
                raise RefcountError("sharing a block that is free")
        for p in ids:
            self.ref[p] += 1
            self.ext[p] += 1

    def cow(self, p: int) -> int:
        """Make the caller's handle on ``p`` private.  Returns the block the
        caller should write (``p`` itself when it is not shared)."""
        self._check_ids([p])
        if self.ext[p] < 1:
            raise RefcountError("copy-on-write of a handle that is not held")
        if self.ref[p] == 1:
            return p
        new = self._pop_free()
        self.ref[p] -= 1
        self.ext[p] -= 1
        self.ref[new] = 1
        self.ext[new] = 1
        return new

    # ------------------------------------------------------------------
    # views and checks
    # ------------------------------------------------------------------
    def stats(self):
        n_free = len(self.free)
        n_shared = sum(1 for c in self.ref if c > 1)
        return n_free, self.num_blocks - n_free, n_shared

    def block_table(self, seq_ids, max_blocks: int):
        """Rows padded with -1, plus the context lengths."""
        rows, lens = [], []
        for s in seq_ids:
            t = self.tables.get(s, [])
            if len(t) > max_blocks:
                raise InvalidArg("table wider than max_blocks")
            rows.append(list(t) + [-1] * (max_blocks - len(t)))
            lens.append(self.lengths.get(s, 0))
        return rows, lens

    def check(self) -> None:
        """The conservation checks of §13, plus ``ref = table refs + handles``."""
        n_free = len(self.free)
        assert len(set(self.free)) == n_free, "duplicate id on the free list"
        allocated = set(range(self.num_blocks)) - set(self.free)
        assert n_free + len(allocated) == self.num_blocks
        assert {p for p in range(self.num_blocks) if self.ref[p] > 0} == allocated
        table_refs = [0] * self.num_blocks
        for s, t in self.tables.items():
            assert len(t) == -(-self.lengths[s] // self.block_size)
            for p in t:
                table_refs[p] += 1
        for p in range(self.num_blocks):
            assert self.ref[p] == table_refs[p] + self.ext[p]
