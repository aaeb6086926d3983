"""Oracle block manager: physical blocks, block tables, reference counts, CoW.

Test infrastructure (see the package docstring). Plain Python, one token at a time.

Sources:
- vLLM docs page (docs.acceleratez.fun, "vLLM"), section PagedAttention ›
  算法流程 (algorithm flow): prefill splits the prompt into blocks of B tokens;
  in decode, after each new token, check whether the current block is full and
  only then allocate a new physical block and extend the block table; when a
  request finishes, release all its blocks.
- Same page, section 显存利用率分析: a request of n tokens holds ceil(n/B) blocks.
- Same page, section Copy-on-Write › 引用计数管理 (ref counts): a sharer adds 1,
  a finished request subtracts 1 from every block of its table, a block whose
  count reaches 0 is released.
- Same page, Copy-on-Write › 写时复制: when a request writes into a block whose
  count is > 1, allocate a new block, copy the old block into it, write the
  token there, point the table at the new block and subtract 1 from the old one.
- vLLM code-reading page (sourceaix.com), §5.1.1 单个请求 (the 7-token prompt,
  B = 4, physical blocks 7 and 1) and §5.2.1 Parallel Sampling (A1/A2 share
  blocks 7/1 with ref count 2; A1's divergent write moves it to block 3).
- vLLM 0.10.0 flow page (ascendai.csdn.net), §3.3 KV Manager模块: a slot is one
  token's position, slot = physical_block * B + offset.

Readings where the pages leave a choice open:
- Free blocks are handed out first-in first-out from an explicit initial order;
  a released block goes to the tail of that queue.
- Allocation is lazy: a block is taken only when a token must be written and the
  last block is full (or the table is empty).
- Among the sharers of a block, whichever writes while the count is > 1 copies;
  the last remaining holder writes in place.
- An append that cannot be satisfied changes nothing and raises: NoFreeBlocks
  when the free queue is too short right now, TooLarge when the sequence would
  need more blocks than the whole pool.
"""
from __future__ import annotations

from collections import deque


class NoFreeBlocks(RuntimeError):
    """Not enough free blocks now (the request could run later)."""


class TooLarge(RuntimeError):
    """The sequence would need more blocks than the pool holds."""


class BlockAllocator:
    def __init__(self, num_blocks: int, block_size: int, free_order):
        free_order = [int(b) for b in free_order]
        if sorted(free_order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of range(num_blocks)")
        self.num_blocks = num_blocks
        self.B = block_size
        self.free = deque(free_order)
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}
        self.pending_copies: list[tuple[int, int]] = []

    # -- queries ---------------------------------------------------------
    def block_table(self, seq: int) -> list[int]:
        return list(self.tables[seq])

    def seq_len(self, seq: int) -> int:
        return self.lens[seq]

    def ref_count(self, block: int) -> int:
        return self.ref[block]

    def num_free(self) -> int:
        return len(self.free)

    def filled(self, seq: int) -> list[int]:
        """The '# filled' column of the block table: tokens held by each logical block."""
        n, out = self.lens[seq], []
        for _ in self.tables[seq]:
            out.append(min(self.B, n))
            n -= min(self.B, n)
        return out

    # -- operations --------------------------------------------------------
    def add_seq(self, seq: int) -> None:
        if seq in self.tables:
            raise ValueError(f"sequence {seq} exists")
        self.tables[seq] = []
        self.lens[seq] = 0

    def _pop(self) -> int:
        b = self.free.popleft()
        self.ref[b] = 1
        return b

    def blocks_needed(self, seq: int, n: int) -> int:
        """Free blocks an append of n tokens would take from the queue."""
        L, table = self.lens[seq], self.tables[seq]
        if n <= 0:
            return 0
        new_blocks = -(-(L + n) // self.B) - -(-L // self.B)
        cow = 1 if (L % self.B != 0 and self.ref[table[-1]] > 1) else 0
        return new_blocks + cow

    def append(self, seq: int, n: int) -> list[int]:
        """Append n tokens to ``seq``; returns the slot of each new token."""
        if -(-(self.lens[seq] + n) // self.B) > self.num_blocks:
            raise TooLarge(f"sequence {seq} would need more than {self.num_blocks} blocks")
        if self.blocks_needed(seq, n) > len(self.free):
            raise NoFreeBlocks(f"sequence {seq} needs {self.blocks_needed(seq, n)} blocks, {len(self.free)} free")
        table = self.tables[seq]
        slots = []
        for _ in range(n):
            L = self.lens[seq]
            if L % self.B == 0:
                table.append(self._pop())  # last block full (or none yet): take a new one
            elif self.ref[table[-1]] > 1:
                old = table[-1]  # shared partial block: copy before writing
                new = self._pop()
                self.pending_copies.append((old, new))
                table[-1] = new
                self.ref[old] -= 1
            slots.append(table[L // self.B] * self.B + L % self.B)
            self.lens[seq] = L + 1
        return slots

    def fork(self, parent: int, child: int) -> None:
        """``child`` starts with ``parent``'s blocks, shared (each count + 1)."""
        if child in self.tables:
            raise ValueError(f"sequence {child} exists")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def free_seq(self, seq: int) -> None:
        """Release ``seq``: every block's count - 1; blocks reaching 0 rejoin the queue tail."""
        for b in self.tables.pop(seq):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
            elif self.ref[b] < 0:
                raise AssertionError("negative reference count")
        del self.lens[seq]

    def take_copies(self) -> list[tuple[int, int]]:
        """CoW (src, dst) pairs emitted since the last call, in emission order."""
        out, self.pending_copies = self.pending_copies, []
        return out
