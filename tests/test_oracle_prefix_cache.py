"""Pins of the oracle's prefix caching (CPU only).

- The memory-saving table of the vLLM docs page (Copy-on-Write › 优势分析: 10 requests
  with one system prompt keep 1 copy of the prefix KV instead of 10, a 90 % saving;
  100 requests, 99 %), as a closed form over block counts.
- A shadow model of slot contents, independent of the allocator's keys: every reused
  prefix reads back, through the block table, exactly the prompt tokens it stands for,
  and every registered block holds the prefix it is registered under.
- Scenarios fixing each reading: reuse after release, LRU eviction order, the walk
  stopping at the first miss, the first registration winning, the last prompt token
  never reused, reuse of a block still held by a live request.
"""
import random

import pytest

from oracle import BlockAllocator, PrefixCachingAllocator


def _prompt_run(alloc, seq, prompt, cached=True):
    """Admit ``seq`` with ``prompt``: reuse what is cached, append the rest. Returns hit."""
    if cached:
        hit = alloc.add_seq_cached(seq, prompt, max_hit=len(prompt) - 1)
        alloc.append(seq, len(prompt) - hit, tokens=prompt[hit:])
        return hit
    alloc.add_seq(seq)
    alloc.append(seq, len(prompt))
    return 0


@pytest.mark.parametrize("R,saving", [(10, 0.90), (100, 0.99)])
def test_shared_system_prompt_saving_matches_the_page(R, saving):
    B, P = 16, 256
    system = list(range(1000, 1000 + P))
    NB = 4096
    order = list(range(NB))
    c, u = PrefixCachingAllocator(NB, B, order), BlockAllocator(NB, B, order)
    for r in range(R):
        prompt = system + [r]  # one private token after the shared prompt
        hit = _prompt_run(c, r, prompt)
        _prompt_run(u, r, prompt, cached=False)
        assert hit == (0 if r == 0 else P)
    prefix_blocks = P // B
    held_c = {b for r in range(R) for b in c.block_table(r)[:prefix_blocks]}
    held_u = {b for r in range(R) for b in u.block_table(r)[:prefix_blocks]}
    assert len(held_c) == prefix_blocks and len(held_u) == R * prefix_blocks
    assert abs((len(held_u) - len(held_c)) / len(held_u) - saving) < 1e-12
    for b in held_c:
        assert c.ref_count(b) == R
    assert NB - c.num_free() == prefix_blocks + R  # + one private block per request


class Shadow:
    """Token id stored in every slot, updated from slots and copy pairs only."""

    def __init__(self, alloc):
        self.a = alloc
        self.content = {}

    def write(self, slots, tokens):
        for s, t in zip(slots, tokens):
            self.content[s] = t

    def copies(self):
        B = self.a.B
        for src, dst in self.a.take_copies():
            for o in range(B):
                if src * B + o in self.content:
                    self.content[dst * B + o] = self.content[src * B + o]
                else:
                    self.content.pop(dst * B + o, None)

    def logical(self, seq):
        B, table = self.a.B, self.a.block_table(seq)
        return [self.content.get(table[p // B] * B + p % B) for p in range(self.a.seq_len(seq))]

    def check(self):
        a, B = self.a, self.a.B
        for key, b in a.cached.items():
            assert len(key) % B == 0
            assert [self.content.get(b * B + o) for o in range(B)] == list(key[-B:])
            assert a.key_of[b] == key
        for seq in a.tables:
            toks = self.logical(seq)
            assert toks == a.tokens[seq]
            for i, b in enumerate(a.block_table(seq)):
                if b in a.key_of and (i + 1) * B <= len(toks):
                    assert a.key_of[b] == tuple(toks[: (i + 1) * B])
        held = [b for t in a.tables.values() for b in t]
        for b in range(a.num_blocks):
            assert a.ref_count(b) == held.count(b)
            assert (b in a.free) == (a.ref_count(b) == 0)


@pytest.mark.parametrize("seed", range(12))
def test_random_operations_keep_keys_true_to_content(seed):
    rng = random.Random(seed)
    B = rng.choice([1, 2, 4, 8])
    NB = rng.randint(8, 40)
    order = list(range(NB))
    rng.shuffle(order)
    a = PrefixCachingAllocator(NB, B, order)
    sh = Shadow(a)
    bases = [[rng.randint(0, 3) for _ in range(rng.randint(0, 4 * B))] for _ in range(3)]
    live, nxt, hits = [], 0, 0
    for _ in range(300):
        op = rng.random()
        try:
            if op < 0.3 or not live:
                prompt = list(rng.choice(bases)) + [rng.randint(0, 3) for _ in range(rng.randint(1, 2 * B))]
                s = nxt
                nxt += 1
                hit = a.add_seq_cached(s, prompt, max_hit=len(prompt) - 1)
                live.append(s)
                hits += hit
                assert sh.logical(s) == prompt[:hit]  # a reused prefix holds exactly these tokens
                slots = a.append(s, len(prompt) - hit, tokens=prompt[hit:])
                sh.copies()
                sh.write(slots, prompt[hit:])
            elif op < 0.6:
                s = rng.choice(live)
                toks = [rng.randint(0, 3) for _ in range(rng.randint(1, B + 1))]
                slots = a.append(s, len(toks), tokens=toks)
                sh.copies()
                sh.write(slots, toks)
            elif op < 0.75:
                a.fork(rng.choice(live), nxt)
                live.append(nxt)
                nxt += 1
            else:
                s = rng.choice(live)
                a.free_seq(s)
                live.remove(s)
        except Exception as e:  # a pool too small for this append: it changed nothing
            assert type(e).__name__ in ("NoFreeBlocks", "TooLarge"), e
        sh.check()
    assert hits > 0


def _fill(a, seq, tokens):
    a.add_seq(seq)
    return a.append(seq, len(tokens), tokens=tokens)


def test_reuse_after_release_takes_the_same_blocks_out_of_the_queue():
    B = 4
    a = PrefixCachingAllocator(16, B, list(range(16)))
    p = list(range(14))  # 3 full blocks + 2 tokens
    _fill(a, 0, p)
    first = a.block_table(0)
    a.free_seq(0)
    assert a.num_free() == 16 and a.num_cached() == 3
    hit = a.add_seq_cached(1, p + [99], max_hit=14)
    assert hit == 12
    assert a.block_table(1) == first[:3]
    assert a.num_free() == 13 and all(a.ref_count(b) == 1 for b in first[:3])
    assert list(a.free)[-1] == first[3]  # the partial block was released, not reused


def test_lru_eviction_and_walk_stops_at_first_miss():
    B = 4
    a = PrefixCachingAllocator(8, B, list(range(8)))
    p = list(range(12))  # exactly 3 full blocks: 0, 1, 2
    _fill(a, 0, p)
    assert a.block_table(0) == [0, 1, 2]
    a.free_seq(0)  # queue: 3 4 5 6 7 0 1 2
    _fill(a, 1, list(range(100, 100 + 6 * B)))  # takes 3..7 and then 0: block 0 evicted
    assert a.block_table(1) == [3, 4, 5, 6, 7, 0]
    assert a.evictions == 1 and a.num_cached() == 2 + 6  # blocks 1, 2 still cached; 6 new
    hit = a.add_seq_cached(2, p + [7], max_hit=12)
    assert hit == 0  # the walk stops at the evicted first block


def test_first_registration_wins_and_last_token_is_never_reused():
    B = 4
    a = PrefixCachingAllocator(16, B, list(range(16)))
    p = list(range(8))
    a.add_seq(0)
    a.add_seq(1)
    a.append(0, 8, tokens=p)  # registers blocks 0, 1
    a.append(1, 8, tokens=p)  # same prefix computed again: blocks 2, 3 stay private
    assert a.cached == {tuple(p[:4]): 0, tuple(p): 1}
    a.free_seq(1)
    a.free_seq(0)
    hit = a.add_seq_cached(2, p, max_hit=len(p) - 1)
    assert hit == 4 and a.block_table(2) == [0]  # block 1 would cover the last token


def test_reuse_of_a_block_held_by_a_live_request():
    B = 4
    a = PrefixCachingAllocator(16, B, list(range(16)))
    p = list(range(9))
    _fill(a, 0, p)  # blocks 0, 1 full, 2 partial
    hit = a.add_seq_cached(1, p[:8] + [50, 51], max_hit=9)
    assert hit == 8 and a.block_table(1) == [0, 1]
    assert a.ref_count(0) == 2 and a.ref_count(1) == 2
    slots = a.append(1, 2, tokens=[50, 51])
    assert slots == [3 * B, 3 * B + 1] and a.take_copies() == []  # a fresh block, no copy
