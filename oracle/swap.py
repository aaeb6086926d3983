"""Oracle swapping: preempted requests' blocks moved to a CPU block pool and back.

Test infrastructure (see the package docstring). Plain Python.

Sources:
- vLLM code-reading page (sourceaix.com), §6.2.1 SequenceGroup: when the GPU runs out of
  resources the scheduler preempts a sequence group; with more than one sequence its KV
  blocks are swapped out to the CPU (status swapped), with one sequence they are freed and
  the request is recomputed later; when resources return the CPU blocks are swapped back
  in and the group runs again.
- VLLM overview page (dn008.com.cn), §4 scheduler structure › scheduling flow › swap
  phase: under resource pressure lower-priority work moves to CPU memory (the swapped
  queue), like page swapping in an OS.
- vLLM docs page (docs.acceleratez.fun, "vLLM"), Copy-on-Write › reference counts
  (a block is held by several sequences; it is released when its count reaches 0).

Readings where the pages leave a choice open (the plainest ones):
- The CPU pool works like the GPU pool: its own blocks, a FIFO free queue from a given
  order, reference counts.
- A swap moves a set of sequences together (a group). Each distinct block their tables
  hold is copied once, to one new block on the other side, in the order first met walking
  the sequences in the given order and each table from its first block. The new block's
  count is the number of those sequences holding it; the old block's count drops by the
  same number and the block is released at 0 (a block still held by others stays).
- A swap that does not fit the other pool changes nothing. A swapped sequence takes no
  appends or forks until it is swapped back in; ending it releases its CPU blocks.
- Blocks arriving on the GPU are ordinary private blocks (no prefix-cache registration).
"""
from __future__ import annotations

from collections import deque

from .block_manager import BlockAllocator, NoFreeBlocks
from .prefix_cache import PrefixCachingAllocator


class SwapMixin:
    """Adds a CPU block pool and swap_out / swap_in to an allocator."""

    def enable_swap(self, num_cpu_blocks: int, cpu_free_order):
        order = [int(b) for b in cpu_free_order]
        if sorted(order) != list(range(num_cpu_blocks)):
            raise ValueError("cpu_free_order must be a permutation of range(num_cpu_blocks)")
        self.num_cpu_blocks = num_cpu_blocks
        self.cpu_free = deque(order)
        self.cpu_ref = [0] * num_cpu_blocks
        self.swapped: set = set()

    def _group_blocks(self, seqs):
        """Distinct blocks of the group's tables in first-met order, with their holder counts."""
        order, holders = [], {}
        for s in seqs:
            for b in self.tables[s]:
                if b not in holders:
                    holders[b] = 0
                    order.append(b)
                holders[b] += 1
        return order, holders

    def swap_out(self, seqs) -> list[tuple[int, int]]:
        """Move the group's blocks GPU -> CPU; returns the (gpu block, cpu block) copies."""
        seqs = list(seqs)
        if len(set(seqs)) != len(seqs) or any(s not in self.tables or s in self.swapped for s in seqs):
            raise ValueError("swap_out takes distinct sequences resident on the GPU")
        order, holders = self._group_blocks(seqs)
        if len(order) > len(self.cpu_free):
            raise NoFreeBlocks(f"swap out needs {len(order)} CPU blocks, {len(self.cpu_free)} free")
        where, pairs = {}, []
        for g in order:
            c = self.cpu_free.popleft()
            self.cpu_ref[c] = holders[g]
            self.ref[g] -= holders[g]
            if self.ref[g] == 0:
                self.free.append(g)
            where[g] = c
            pairs.append((g, c))
        for s in seqs:
            self.tables[s] = [where[b] for b in self.tables[s]]
            self.swapped.add(s)
        return pairs

    def swap_in(self, seqs) -> list[tuple[int, int]]:
        """Move the group's blocks CPU -> GPU; returns the (cpu block, gpu block) copies."""
        seqs = list(seqs)
        if len(set(seqs)) != len(seqs) or any(s not in self.swapped for s in seqs):
            raise ValueError("swap_in takes distinct swapped sequences")
        order, holders = self._group_blocks(seqs)
        if len(order) > len(self.free):
            raise NoFreeBlocks(f"swap in needs {len(order)} GPU blocks, {len(self.free)} free")
        where, pairs = {}, []
        for c in order:
            g = self._pop()
            self.ref[g] = holders[c]
            self.cpu_ref[c] -= holders[c]
            if self.cpu_ref[c] == 0:
                self.cpu_free.append(c)
            where[c] = g
            pairs.append((c, g))
        for s in seqs:
            self.tables[s] = [where[b] for b in self.tables[s]]
            self.swapped.discard(s)
        return pairs

    # a swapped sequence is frozen; ending it releases CPU blocks
    def append(self, seq, n, *args, **kw):
        if seq in getattr(self, "swapped", ()):
            raise ValueError(f"sequence {seq} is swapped out")
        return super().append(seq, n, *args, **kw)

    def fork(self, parent, child):
        if parent in getattr(self, "swapped", ()):
            raise ValueError(f"sequence {parent} is swapped out")
        return super().fork(parent, child)

    def free_seq(self, seq):
        if seq in getattr(self, "swapped", ()):
            for c in self.tables.pop(seq):
                self.cpu_ref[c] -= 1
                if self.cpu_ref[c] == 0:
                    self.cpu_free.append(c)
            del self.lens[seq]
            if hasattr(self, "tokens"):
                del self.tokens[seq]
            self.swapped.discard(seq)
            return
        super().free_seq(seq)


class SwappingAllocator(SwapMixin, BlockAllocator):
    pass


class SwappingPrefixAllocator(SwapMixin, PrefixCachingAllocator):
    pass
