"""Pins of the oracle block manager against what the pages fix (CPU only)."""
import json
import math
import os
import random

import pytest

from oracle import BlockAllocator, NoFreeBlocks, TooLarge

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _order(head, n=16):
    return list(head) + [b for b in range(n) if b not in head]


def test_single_request_worked_example():
    g = _golden("single_request_b4.json")
    a = BlockAllocator(16, g["block_size"], _order(g["free_order_head"]))
    a.add_seq(0)
    slots = a.append(0, g["prompt_tokens"])
    assert a.block_table(0) == g["after_prefill"]["block_table"]
    assert a.filled(0) == g["after_prefill"]["filled"]
    # slots of the prompt: block 7 offsets 0..3, block 1 offsets 0..2
    assert slots == [7 * 4 + i for i in range(4)] + [1 * 4 + i for i in range(3)]
    a.append(0, 1)  # 'fathers'
    assert a.block_table(0) == g["after_first_token"]["block_table"]
    assert a.filled(0) == g["after_first_token"]["filled"]
    a.append(0, 1)
    assert a.block_table(0) == g["after_second_token"]["block_table"]
    assert a.filled(0) == g["after_second_token"]["filled"]


def test_parallel_sampling_cow_example():
    g = _golden("parallel_sampling_cow.json")
    a = BlockAllocator(16, g["block_size"], _order(g["free_order_head"]))
    A1, A2 = 1, 2
    a.add_seq(A1)
    a.append(A1, g["prompt_tokens"])
    a.fork(A1, A2)
    refs = lambda: {str(b): a.ref_count(b) for b in set(a.block_table(A1)) | set(a.block_table(A2))}  # noqa: E731
    assert a.block_table(A1) == g["after_fork"]["A1"] and a.block_table(A2) == g["after_fork"]["A2"]
    assert refs() == g["after_fork"]["ref"]
    s1 = a.append(A1, 1)  # 'fathers'
    assert a.block_table(A1) == g["after_A1_write"]["A1"]
    assert a.block_table(A2) == g["after_A1_write"]["A2"]
    assert refs() == g["after_A1_write"]["ref"]
    assert [list(p) for p in a.take_copies()] == g["after_A1_write"]["copies"]
    assert s1 == [3 * 4 + 3]  # offset 3 of the new block
    s2 = a.append(A2, 1)  # 'mothers': block 1 is now private, written in place
    assert a.block_table(A2) == g["after_A2_write"]["A2"]
    assert refs() == g["after_A2_write"]["ref"]
    assert [list(p) for p in a.take_copies()] == g["after_A2_write"]["copies"]
    assert s2 == [1 * 4 + 3]


def test_memory_arithmetic():
    g = _golden("memory_arithmetic.json")
    a = BlockAllocator(64, g["block_size"], range(64))
    a.add_seq(0)
    a.append(0, g["tokens"])
    assert len(a.block_table(0)) == g["blocks"]
    assert len(a.block_table(0)) * g["block_size"] * g["kv_bytes_per_token"] == g["paged_bytes"]
    assert g["tokens"] * g["kv_bytes_per_token"] / (g["reserved_tokens"] * g["kv_bytes_per_token"]) == \
        g["contiguous_utilisation"]


@pytest.mark.parametrize("B", [1, 4, 16])
def test_lazy_allocation_one_token_at_a_time(B):
    a = BlockAllocator(40, B, range(40))
    a.add_seq(0)
    for n in range(1, 3 * B + 2):
        before = len(a.block_table(0))
        a.append(0, 1)
        after = len(a.block_table(0))
        assert after == math.ceil(n / B)
        # a new block appears exactly when the previous last block was full
        assert (after - before) == (1 if (n - 1) % B == 0 else 0)
        assert a.num_free() == 40 - after


def test_ref_count_lifecycle_and_release_order():
    a = BlockAllocator(8, 4, [5, 2, 7, 0, 1, 3, 4, 6])
    a.add_seq(0)
    a.append(0, 8)  # two full blocks: 5, 2
    for c in (1, 2, 3):
        a.fork(0, c)
    assert [a.ref_count(b) for b in (5, 2)] == [4, 4]
    a.free_seq(1)
    assert [a.ref_count(b) for b in (5, 2)] == [3, 3]
    a.free_seq(0)
    a.free_seq(2)
    assert a.num_free() == 6
    a.free_seq(3)  # counts reach 0: both rejoin the queue tail, in table order
    assert list(a.free)[-2:] == [5, 2]
    assert a.num_free() == 8


def test_fork_of_full_block_takes_new_block_without_copy():
    a = BlockAllocator(8, 4, range(8))
    a.add_seq(0)
    a.append(0, 4)
    a.fork(0, 1)
    a.append(1, 1)
    assert a.take_copies() == []
    assert a.block_table(1) == [0, 1] and a.block_table(0) == [0]
    assert a.ref_count(0) == 2


def test_exhaustion_is_atomic():
    a = BlockAllocator(3, 4, range(3))
    a.add_seq(0)
    a.append(0, 9)  # 3 blocks
    a.add_seq(1)
    with pytest.raises(NoFreeBlocks):
        a.append(1, 1)
    assert a.block_table(1) == [] and a.seq_len(1) == 0
    with pytest.raises(TooLarge):
        a.append(0, 4)  # would need 4 blocks in a pool of 3
    assert a.seq_len(0) == 9 and a.block_table(0) == [0, 1, 2]
    a.fork(0, 2)
    with pytest.raises(NoFreeBlocks):
        a.append(2, 1)  # the CoW copy needs a free block
    assert a.block_table(2) == [0, 1, 2] and a.take_copies() == []


def _check_invariants(a, live_lens):
    holders = {}
    for s, t in a.tables.items():
        assert len(t) == math.ceil(a.seq_len(s) / a.B)
        assert a.seq_len(s) == live_lens[s]
        for b in t:
            holders[b] = holders.get(b, 0) + 1
    for b in range(a.num_blocks):
        assert a.ref_count(b) == holders.get(b, 0)
    assert a.num_free() + len(holders) == a.num_blocks
    assert set(a.free).isdisjoint(holders)
    assert len(set(a.free)) == a.num_free()


@pytest.mark.parametrize("seed", range(20))
def test_random_operation_sequences_keep_invariants(seed):
    rng = random.Random(seed)
    B = rng.choice([1, 2, 4, 16])
    N = rng.randint(4, 40)
    a = BlockAllocator(N, B, rng.sample(range(N), N))
    lens, nxt = {}, 0
    for _ in range(200):
        op = rng.random()
        if op < 0.2 or not lens:
            a.add_seq(nxt)
            lens[nxt] = 0
            nxt += 1
        elif op < 0.6:
            s = rng.choice(list(lens))
            n = rng.randint(0, 2 * B + 1)
            shared_before = bool(a.tables[s]) and a.ref_count(a.tables[s][-1]) > 1 and lens[s] % B != 0
            try:
                free_before = a.num_free()
                slots = a.append(s, n)
            except (NoFreeBlocks, TooLarge):
                assert a.num_free() == free_before
            else:
                copies = a.take_copies()
                assert len(copies) == (1 if (shared_before and n > 0) else 0)
                for src, dst in copies:
                    assert a.ref_count(dst) == 1 and dst == a.tables[s][(lens[s]) // B]
                for i, slot in enumerate(slots):
                    p = lens[s] + i
                    assert slot == a.tables[s][p // B] * B + p % B
                lens[s] += n
        elif op < 0.8:
            p = rng.choice(list(lens))
            a.fork(p, nxt)
            lens[nxt] = lens[p]
            nxt += 1
        else:
            s = rng.choice(list(lens))
            a.free_seq(s)
            del lens[s]
        _check_invariants(a, lens)
