"""Oracle prefix cache: full-block prefix reuse across requests with
block-aligned truncation and leaf-first LRU eviction.
TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources, by page title and section:

* "KV 缓存管理", radix-tree section (Table 2, "最长前缀匹配") -- a prefix index
  binds token slices to ordered physical block ids; a new prompt is matched
  from the root, slice by slice, until a token differs or the prompt ends:
  the longest matching path.
* same section, block-boundary problem -- only completely filled blocks are
  shared between requests; the usable hit is rounded down to a whole block,
  ``S_usable = floor(S_match / B) * B``, and the ``S_match mod B`` tail tokens
  are treated as misses and prefilled with the new suffix (block-aligned
  truncation, the strategy the pages prefer to copying the tail).
* same section, the rolling chain ``h_k = Hash(h_{k-1} || c_k)`` over
  16-token chunks -- a chunk's identity is the whole prefix up to its end;
  "第 11 章 KV Cache 内存管理" §11.5 -- the cache key must include everything
  that changes the KV numbers (model, template, adapters ...): here a caller
  ``salt`` that starts the chain.
* same section, "动态基数树淘汰" -- a node referenced by running requests
  (``ref_count >= 1``) is pinned; at ``ref_count = 0`` it is dormant, kept for
  reuse; eviction frees the least recently used dormant *leaf* first
  (a parent is never evicted while a child is cached); when a parent loses
  its last child and is itself dormant it becomes a candidate.

This oracle keeps the cache at block granularity: a cached node is one full
physical block, identified exactly by ``(salt, tokens 0 .. (k+1)B - 1)``
(a tuple, so no hash collision can alias two prefixes).  Readings where the
pages leave a step open:

* A block is published when it fills, at the end of the append call that
  filled it, iff its key is not cached yet and it is the first block of its
  table or the block before it in the same table is a cached node (so every
  cached node's parent is cached).  A block whose content duplicates a cached
  key stays private.
* A new sequence matches once, before its first append (``match_prefix``);
  its tokens past the match are appended and prefilled as usual.
* Eviction runs when a block is needed and the free list is empty (one leaf
  per missing block), or on request (``evict(target_free)``, the pages'
  low-water-mark round).
* ``last_access`` is a logical clock; every node a call touches gets the next
  tick, in table order: the blocks a match takes, a block being published,
  a block that becomes dormant.
"""

from __future__ import annotations

from .block_manager import BlockManager, InvalidArg, NoFreeBlock


class PrefixCachingBlockManager(BlockManager):
    def __init__(self, num_blocks: int, block_size: int, free_order=None, salt: int = 0):
        super().__init__(num_blocks, block_size, free_order)
        self.salt = int(salt)
        self.tokens: dict[int, list] = {}   # per sequence: token ids (None = unknown)
        self.index: dict[tuple, int] = {}   # prefix key -> cached block
        self.key_of: dict[int, tuple] = {}  # cached block -> its key
        self.children: dict[int, int] = {}  # cached block -> number of cached children
        self.last: dict[int, int] = {}      # cached block -> last access tick
        self.dormant: set[int] = set()      # cached blocks with count 0
        self.clock = 0

    # ------------------------------------------------------------- helpers
    def _tick(self, p: int) -> None:
        self.clock += 1
        self.last[p] = self.clock

    def _key(self, toks, k: int):
        """Key of block k of a token list (None while a token is unknown)."""
        part = toks[: (k + 1) * self.block_size]
        if len(part) < (k + 1) * self.block_size or any(t is None for t in part):
            return None
        return (self.salt,) + tuple(part)

    def _leaf_candidates(self):
        return [p for p in self.dormant if self.children.get(p, 0) == 0]

    def _evict_one(self) -> bool:
        cands = self._leaf_candidates()
        if not cands:
            return False
        p = min(cands, key=lambda b: self.last[b])
        key = self.key_of.pop(p)
        del self.index[key]
        self.dormant.discard(p)
        self.children.pop(p, None)
        self.last.pop(p, None)
        parent_key = key[:-self.block_size] if len(key) > 1 + self.block_size else None
        if parent_key is not None:
            q = self.index[parent_key]
            self.children[q] -= 1
        self.free.append(p)
        return True

    def _pop_free(self) -> int:
        if not self.free and not self._evict_one():
            raise NoFreeBlock("no free KV block")
        return self.free.popleft()

    def _publish(self, seq: int, first_full: int) -> None:
        """Publish the blocks of ``seq`` from index ``first_full`` on that are
        full now, in table order."""
        table = self.tables.get(seq, [])
        toks = self.tokens.get(seq, [])
        n_full = self.lengths.get(seq, 0) // self.block_size
        for k in range(first_full, n_full):
            p = table[k]
            if p in self.key_of:
                continue
            key = self._key(toks, k)
            if key is None or key in self.index:
                continue
            if k > 0 and table[k - 1] not in self.key_of:
                continue
            self.index[key] = p
            self.key_of[p] = key
            self.children[p] = 0
            if k > 0:
                self.children[table[k - 1]] += 1
            self._tick(p)

    def _snapshot(self):
        import copy

        return (super()._snapshot(),
                copy.deepcopy((self.tokens, self.index, self.key_of, self.children, self.last,
                               self.dormant, self.clock)))

    def _restore(self, snap):
        base, mine = snap
        super()._restore(base)
        (self.tokens, self.index, self.key_of, self.children, self.last, self.dormant,
         self.clock) = mine

    # ----------------------------------------------------------- interface
    def match_prefix(self, seq: int, tokens) -> int:
        """Longest cached chain of full blocks for a new sequence's prompt;
        the sequence starts with those blocks.  Returns the matched token
        count, a multiple of B (block-aligned truncation)."""
        seq = int(seq)
        if seq in self.lengths or seq in self.tables:
            raise InvalidArg("match_prefix needs a new sequence")
        toks = [int(t) for t in tokens]
        blocks = []
        for k in range(len(toks) // self.block_size):
            p = self.index.get(self._key(toks, k))
            if p is None:
                break
            blocks.append(p)
        for p in blocks:
            self.ref[p] += 1
            self.dormant.discard(p)
            self._tick(p)
        n = len(blocks) * self.block_size
        self.tables[seq] = blocks
        self.lengths[seq] = n
        self.tokens[seq] = toks[:n]
        return n

    def append_tokens(self, seq: int, n: int, token_ids=None):
        seq = int(seq)
        first_full = self.lengths.get(seq, 0) // self.block_size
        snap = self._snapshot()
        try:
            slots, cows = super().append_tokens(seq, n)
        except NoFreeBlock:
            self._restore(snap)
            raise
        ids = [None] * n if token_ids is None else [int(t) for t in token_ids]
        if len(ids) != n:
            self._restore(snap)
            raise InvalidArg("token_ids length")
        self.tokens.setdefault(seq, []).extend(ids)
        self._publish(seq, first_full)
        return slots, cows

    def append_slots(self, seq_ids, token_ids=None):
        seq_ids = [int(s) for s in seq_ids]
        firsts = {s: self.lengths.get(s, 0) // self.block_size for s in seq_ids}
        snap = self._snapshot()
        try:
            slots, cows = super().append_slots(seq_ids)
        except NoFreeBlock:
            self._restore(snap)
            raise
        ids = [None] * len(seq_ids) if token_ids is None else [int(t) for t in token_ids]
        for s, t in zip(seq_ids, ids):
            self.tokens.setdefault(s, []).append(t)
        for s in seq_ids:
            self._publish(s, firsts[s])
        return slots, cows

    def fork(self, parent: int, child: int) -> None:
        super().fork(parent, child)
        self.tokens[child] = list(self.tokens.get(parent, []))

    def release(self, seq: int) -> None:
        seq = int(seq)
        if seq not in self.lengths:
            raise InvalidArg("unknown sequence")
        for p in self.tables.pop(seq, []):
            self.ref[p] -= 1
            if self.ref[p] == 0:
                if p in self.key_of:
                    self.dormant.add(p)
                    self._tick(p)
                else:
                    self.free.append(p)
        self.lengths.pop(seq)
        self.tokens.pop(seq, None)

    def evict(self, target_free: int) -> int:
        """Evict dormant leaves, least recently used first, until the free
        list holds ``target_free`` blocks or nothing is evictable."""
        n = 0
        while len(self.free) < target_free and self._evict_one():
            n += 1
        return n

    def check(self) -> None:
        """Conservation with the cache: every block is exactly one of free,
        referenced (count > 0) or dormant (cached, count 0); counts equal the
        table entries plus caller handles; the cache is a tree."""
        super_free = set(self.free)
        for p in range(self.num_blocks):
            states = (p in super_free) + (self.ref[p] > 0) + (p in self.dormant)
            if states != 1:
                raise AssertionError(f"block {p} in {states} states")
        for p in self.dormant:
            assert p in self.key_of and self.ref[p] == 0
        for p, key in self.key_of.items():
            assert self.index[key] == p
            if len(key) > 1 + self.block_size:
                assert key[:-self.block_size] in self.index
        for p in self.key_of:
            kids = sum(1 for q, kq in self.key_of.items()
                       if len(kq) == len(self.key_of[p]) + self.block_size
                       and kq[:len(self.key_of[p])] == self.key_of[p])
            assert kids == self.children[p]
        count = [0] * self.num_blocks
        for t in self.tables.values():
            for p in t:
                count[p] += 1
        for p in range(self.num_blocks):
            assert count[p] + self.ext[p] == self.ref[p]

    def free_blocks(self, ids) -> None:
        """Caller handles: a cached block whose count reaches zero turns
        dormant instead of free."""
        before = len(self.free)
        super().free_blocks(ids)
        added = [self.free.pop() for _ in range(len(self.free) - before)][::-1]
        for p in added:
            if p in self.key_of:
                self.dormant.add(p)
                self._tick(p)
            else:
                self.free.append(p)

    def cache_stats(self):
        """(free, referenced, dormant, cached) block counts."""
        return len(self.free), sum(1 for r in self.ref if r > 0), len(self.dormant), len(self.key_of)
