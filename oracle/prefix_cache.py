"""Oracle prefix caching: full blocks found again by their token prefix, LRU eviction.

Test infrastructure (see the package docstring). Plain Python, one token at a time.

Sources:
- vLLM docs page (docs.acceleratez.fun, "vLLM"), Copy-on-Write › 共享前缀检测
  (a request's prompt prefix is identified by a hash; if that prefix's KV is already
  cached it is reused and the shared blocks' reference counts go up) and
  › 引用计数管理 (+1 per new user of a block, -1 per finished holder, released at 0);
  section Prefix Caching › 实现机制 (hash the prefix, keep computed prefix KV in a
  shared pool, look it up when a request arrives: on a hit reuse the KV and skip its
  prefill, on a miss compute it and cache the result).
- vLLM 0.10.0 flow page (ascendai.csdn.net), §3.3 KV Manager模块: the pool's logical
  blocks form a doubly linked list and old data is evicted least recently used first.

Readings where the pages leave a choice open (the plainest ones):
- The unit of reuse is a full block. The key of a full block is the whole token
  prefix that ends with it (tokens 0 .. (i+1)·B - 1 of its sequence): two blocks are
  interchangeable exactly when those prefixes are equal. (The pages hash the prefix;
  a hash is only an encoding of this key.) A partially filled block is never cached.
- A block is registered when its last slot is written. If its key is already
  registered to another block, the first registration stays and this block remains
  private (it is released normally).
- A released block (count 0) keeps its registration and joins the tail of the free
  queue; the queue is the LRU list. A block taken from the head for a new write loses
  its registration (evicted). A lookup that hits a block sitting in the free queue takes
  it out of the queue (count 0 -> 1).
- A lookup walks the prompt's full blocks from the start and stops at the first miss;
  it never covers the prompt's last token (that token's query must still be computed),
  so at most max_hit tokens are reused.
- Token ids are given with every append; the K/V of a cached prefix are never
  written again.
"""
from __future__ import annotations

from collections import OrderedDict

from .block_manager import BlockAllocator, NoFreeBlocks, TooLarge


class _LRUQueue:
    """The free queue as an ordered set: pop the head, push the tail, unlink any member."""

    def __init__(self, items):
        self._d = OrderedDict((int(b), None) for b in items)

    def popleft(self) -> int:
        return self._d.popitem(last=False)[0]

    def append(self, b: int) -> None:
        self._d[int(b)] = None

    def remove(self, b: int) -> None:
        del self._d[int(b)]

    def __contains__(self, b) -> bool:
        return int(b) in self._d

    def __len__(self) -> int:
        return len(self._d)

    def __iter__(self):
        return iter(self._d)


class PrefixCachingAllocator(BlockAllocator):
    def __init__(self, num_blocks: int, block_size: int, free_order):
        super().__init__(num_blocks, block_size, free_order)
        self.free = _LRUQueue(self.free)
        self.tokens: dict[int, list[int]] = {}
        self.cached: dict[tuple, int] = {}  # full token prefix -> block
        self.key_of: dict[int, tuple] = {}  # block -> its registered prefix
        self.hits = 0  # blocks reused by lookups
        self.evictions = 0

    def num_cached(self) -> int:
        return len(self.cached)

    def add_seq(self, seq: int) -> None:
        super().add_seq(seq)
        self.tokens[seq] = []

    def _pop(self) -> int:
        b = self.free.popleft()
        if b in self.key_of:  # evicted: its content is about to be overwritten
            del self.cached[self.key_of.pop(b)]
            self.evictions += 1
        self.ref[b] = 1
        return b

    def add_seq_cached(self, seq: int, prompt, max_hit: int) -> int:
        """Start ``seq`` from the longest cached prefix of ``prompt`` (whole blocks, at most
        ``max_hit`` tokens). Returns the number of tokens reused."""
        self.add_seq(seq)
        prompt = [int(t) for t in prompt]
        B, table, hit = self.B, self.tables[seq], 0
        while hit + B <= min(max_hit, len(prompt)):
            b = self.cached.get(tuple(prompt[: hit + B]))
            if b is None:
                break
            if self.ref[b] == 0:
                self.free.remove(b)
            self.ref[b] += 1
            table.append(b)
            hit += B
        self.hits += hit // B
        self.lens[seq] = hit
        self.tokens[seq] = prompt[:hit]
        return hit

    def append(self, seq: int, n: int, tokens=None) -> list[int]:
        """Append n tokens (ids ``tokens``) to ``seq``; returns their slots. Each block that
        fills up is registered under its prefix unless that prefix is registered already."""
        if tokens is None or len(tokens) != n:
            raise ValueError("prefix caching needs the id of every appended token")
        if -(-(self.lens[seq] + n) // self.B) > self.num_blocks:
            raise TooLarge(f"sequence {seq} would need more than {self.num_blocks} blocks")
        if self.blocks_needed(seq, n) > len(self.free):
            raise NoFreeBlocks(f"sequence {seq} needs {self.blocks_needed(seq, n)} blocks, {len(self.free)} free")
        B, table, toks = self.B, self.tables[seq], self.tokens[seq]
        slots = []
        for t in tokens:
            L = self.lens[seq]
            if L % B == 0:
                table.append(self._pop())
            elif self.ref[table[-1]] > 1:
                old, new = table[-1], self._pop()
                self.pending_copies.append((old, new))
                table[-1] = new
                self.ref[old] -= 1
            slots.append(table[L // B] * B + L % B)
            toks.append(int(t))
            self.lens[seq] = L + 1
            if (L + 1) % B == 0:
                key = tuple(toks)
                if key not in self.cached:
                    self.cached[key] = table[-1]
                    self.key_of[table[-1]] = key
        return slots

    def fork(self, parent: int, child: int) -> None:
        super().fork(parent, child)
        self.tokens[child] = list(self.tokens[parent])

    def free_seq(self, seq: int) -> None:
        super().free_seq(seq)
        del self.tokens[seq]
