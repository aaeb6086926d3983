"""Pins of the oracle's swapping (CPU only).

- The code-reading page's SequenceGroup lifecycle (§6.2.1): a 4-sample group is preempted
  (its KV blocks swapped out to the CPU), the GPU blocks are reused by other work, and the
  group is swapped back in and continues, reading exactly the tokens it had.
- A shadow model of slot contents in both pools, updated only from the emitted copy pairs
  and the appends' slots, over random scripts with forks, copy-on-write, releases and
  swaps: every live sequence always reads back its own token stream; reference counts
  equal holders in each pool; no block is lost or double-freed.
- Group rules: a block shared inside the group is copied once; a block also held outside
  the group stays on the GPU; a swap that does not fit changes nothing.
"""
import random

import pytest

from oracle import NoFreeBlocks
from oracle.swap import SwappingAllocator, SwappingPrefixAllocator


class Pools:
    """Token id per (pool, slot), from appends and copies only."""

    def __init__(self, a):
        self.a = a
        self.c = {}

    def write(self, slots, toks):
        for s, t in zip(slots, toks):
            self.c[("g", s)] = t

    def copy(self, pairs, src_pool, dst_pool):
        B = self.a.B
        for src, dst in pairs:
            for o in range(B):
                v = self.c.get((src_pool, src * B + o))
                if v is None:
                    self.c.pop((dst_pool, dst * B + o), None)
                else:
                    self.c[(dst_pool, dst * B + o)] = v

    def cow(self):
        self.copy(self.a.take_copies(), "g", "g")

    def read(self, seq):
        B, pool = self.a.B, ("c" if seq in self.a.swapped else "g")
        t = self.a.tables[seq]
        return [self.c.get((pool, t[p // B] * B + p % B)) for p in range(self.a.lens[seq])]


def _check_counts(a):
    gpu_held = [b for s, t in a.tables.items() if s not in a.swapped for b in t]
    cpu_held = [b for s, t in a.tables.items() if s in a.swapped for b in t]
    for b in range(a.num_blocks):
        assert a.ref[b] == gpu_held.count(b)
        assert (b in a.free) == (a.ref[b] == 0)
    for c in range(a.num_cpu_blocks):
        assert a.cpu_ref[c] == cpu_held.count(c)
        assert (c in a.cpu_free) == (a.cpu_ref[c] == 0)
    assert len(a.free) + len(set(gpu_held)) == a.num_blocks
    assert len(a.cpu_free) + len(set(cpu_held)) == a.num_cpu_blocks


def test_sequence_group_lifecycle_from_the_page():
    B = 4
    a = SwappingAllocator(16, B, list(range(16)))
    a.enable_swap(12, list(range(12)))
    sh = Pools(a)
    prompt = list(range(10))  # 2 full blocks + 2 tokens
    a.add_seq(0)
    sh.write(a.append(0, 10), prompt)
    for i in range(1, 4):
        a.fork(0, i)  # n = 4 samples share the prompt's blocks
    streams = {}
    for i in range(4):
        toks = [100 + 10 * i, 101 + 10 * i, 102 + 10 * i]
        slots = a.append(i, 3)
        sh.cow()
        sh.write(slots, toks)
        streams[i] = prompt + toks
    used_before = 16 - a.num_free()
    pairs = a.swap_out([0, 1, 2, 3])  # preempted: the whole group goes to the CPU
    sh.copy(pairs, "g", "c")
    assert len(pairs) == used_before  # every distinct block once
    assert a.num_free() == 16 and a.swapped == {0, 1, 2, 3}
    for i in range(4):
        assert sh.read(i) == streams[i]
    a.add_seq(9)  # other work reuses the GPU blocks meanwhile
    sh.write(a.append(9, 16 * B - 4), [7] * (16 * B - 4))
    a.free_seq(9)
    pairs = a.swap_in([0, 1, 2, 3])  # resources back: swap in, running again
    sh.copy(pairs, "c", "g")
    assert a.swapped == set() and len(a.cpu_free) == 12
    for i in range(4):
        assert sh.read(i) == streams[i]
    _check_counts(a)
    slots = a.append(2, 1)  # and it continues
    sh.cow()
    sh.write(slots, [999])
    assert sh.read(2) == streams[2] + [999]


def test_partial_group_leaves_shared_blocks_on_the_gpu():
    B = 4
    a = SwappingAllocator(16, B, list(range(16)))
    a.enable_swap(8, list(range(8)))
    a.add_seq(0)
    a.append(0, 8)  # blocks 0, 1 full
    for i in (1, 2, 3):
        a.fork(0, i)
    pairs = a.swap_out([1, 2])
    assert pairs == [(0, 0), (1, 1)]
    assert a.ref_count(0) == 2 and a.ref_count(1) == 2  # 0 and 3 still hold them
    assert a.cpu_ref[0] == 2 and a.cpu_ref[1] == 2
    _check_counts(a)


def test_swap_that_does_not_fit_changes_nothing():
    B = 4
    a = SwappingAllocator(8, B, list(range(8)))
    a.enable_swap(1, [0])
    a.add_seq(0)
    a.append(0, 8)
    with pytest.raises(NoFreeBlocks):
        a.swap_out([0])
    assert a.block_table(0) == [0, 1] and a.swapped == set() and list(a.cpu_free) == [0]
    with pytest.raises(ValueError):
        a.swap_in([0])  # not swapped


@pytest.mark.parametrize("prefix", [False, True])
@pytest.mark.parametrize("seed", range(10))
def test_random_scripts_keep_every_stream(seed, prefix):
    rng = random.Random(seed)
    B = rng.choice([1, 2, 4, 8])
    NB, NC = rng.randint(6, 30), rng.randint(4, 30)
    order, corder = list(range(NB)), list(range(NC))
    rng.shuffle(order)
    rng.shuffle(corder)
    a = (SwappingPrefixAllocator if prefix else SwappingAllocator)(NB, B, order)
    a.enable_swap(NC, corder)
    sh = Pools(a)
    streams, nxt, swaps = {}, 0, 0
    for _ in range(300):
        live = list(streams)
        op = rng.random()
        try:
            if op < 0.2 or not live:
                toks = [rng.randrange(3) for _ in range(rng.randint(1, 3 * B))]
                s, nxt = nxt, nxt + 1
                if prefix:
                    hit = a.add_seq_cached(s, toks, max_hit=len(toks) - 1)
                    streams[s] = toks[:hit]
                    assert sh.read(s) == streams[s]
                    slots = a.append(s, len(toks) - hit, tokens=toks[hit:])
                else:
                    a.add_seq(s)
                    streams[s], hit = [], 0
                    slots = a.append(s, len(toks))
                sh.cow()
                sh.write(slots, toks[hit:])
                streams[s] = toks
            elif op < 0.45:
                s = rng.choice(live)
                toks = [rng.randrange(3) for _ in range(rng.randint(1, B + 1))]
                slots = a.append(s, len(toks), tokens=toks) if prefix else a.append(s, len(toks))
                sh.cow()
                sh.write(slots, toks)
                streams[s] = streams[s] + toks
            elif op < 0.55:
                p = rng.choice(live)
                a.fork(p, nxt)
                streams[nxt] = list(streams[p])
                nxt += 1
            elif op < 0.75:
                group = rng.sample(live, rng.randint(1, min(3, len(live))))
                if all(s in a.swapped for s in group):
                    sh.copy(a.swap_in(group), "c", "g")
                    swaps += 1
                elif not any(s in a.swapped for s in group):
                    sh.copy(a.swap_out(group), "g", "c")
                    swaps += 1
            else:
                s = rng.choice(live)
                a.free_seq(s)
                del streams[s]
        except NoFreeBlocks:
            pass
        except ValueError as e:
            assert "swapped out" in str(e)
        except Exception as e:
            assert type(e).__name__ == "TooLarge", e
        sh.cow()
        for s in streams:
            assert sh.read(s) == streams[s], (s, a.tables[s])
        _check_counts(a)
    assert swaps > 0
