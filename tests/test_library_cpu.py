"""The C-ABI library on a machine without a GPU: it loads, exports every symbol the
header declares, rejects bad arguments before touching CUDA, and its host block manager
agrees exactly with the oracle's (tables, slots, copy pairs, counts, free-queue order)."""
import os
import random
import re

import numpy as np
import pytest

import paged_kv_cache_161_gb300 as pa
import workloads
from oracle import BlockAllocator, NoFreeBlocks, TooLarge, run_allocator

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pa.h")


def _declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", txt)))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert "pa_attention" in names and "pa_kv_write" in names and "pa_copy_blocks" in names
    for n in names:
        assert hasattr(pa.lib, n), n


def test_status_strings():
    assert pa.lib.pa_status_string(0) == b"ok"
    assert b"workspace" in pa.lib.pa_status_string(3)
    assert pa.lib.pa_status_string(12345) == b"unknown status"


def test_bad_arguments_are_rejected_before_any_launch():
    L = pa.lib
    # null caches
    assert L.pa_kv_write(None, None, None, None, None, 1, 8, 16, 8, 128, 1, None) == 1
    # misaligned cache pointer
    assert L.pa_copy_blocks(8, 8, None, 1, 8, 16, 8, 128, 1, None) == 1
    # bad dtype code
    assert L.pa_copy_blocks(16, 16, 16, 1, 8, 16, 8, 128, 7, None) == 1
    # attention: unsupported head_dim, bad group, bad block size
    args = [16, 16, 16, 16, 16, 8, 16, 16, 2, 2, 1, 64, 32, 8, 128, 16, 64, 0.1, 1, 16, 1 << 20, None]
    a = list(args)
    a[14] = 96
    assert L.pa_attention(*a) == 2
    a = list(args)
    a[13] = 3  # 32 query heads over 3 KV heads
    assert L.pa_attention(*a) == 1
    a = list(args)
    a[15] = 24  # block size neither divides nor is a multiple of 16
    assert L.pa_attention(*a) == 2
    a = list(args)
    a[17] = -1.0  # scale
    assert L.pa_attention(*a) == 1
    a = list(args)
    a[5] = 1  # table too narrow for max_seq_len 64 at block size 16
    assert L.pa_attention(*a) == 1
    # the fused write + attention: same checks, plus its write inputs
    wargs = args[:2] + [16, 16, 16] + args[2:]  # k_new, v_new, slot_mapping after q
    for i, val, want in [(17, 96, 2), (16, 3, 1), (18, 24, 2), (20, -1.0, 1), (8, 1, 1),
                         (2, None, 1), (3, 8, 1), (4, 12, 1)]:
        a = list(wargs)
        a[i] = val
        assert L.pa_write_attention(*a) == want, (i, val)


def test_block_manager_rejects_bad_free_order():
    with pytest.raises(ValueError):
        pa.BlockManager(4, 4, [0, 1, 1, 2])
    with pytest.raises(ValueError):
        pa.BlockManager(4, 4, [0, 1, 2, 4])


def _compare(ref: BlockAllocator, bm: pa.BlockManager, seqs):
    for s in seqs:
        assert ref.block_table(s) == bm.block_table(s).tolist()
        assert ref.seq_len(s) == bm.seq_len(s)
    for b in range(ref.num_blocks):
        assert ref.ref_count(b) == bm.ref_count(b)
    assert list(ref.free) == bm.free_queue().tolist()


def test_worked_examples_in_cpp():
    order = [7, 1, 3] + [b for b in range(16) if b not in (7, 1, 3)]
    bm = pa.BlockManager(16, 4, order)
    bm.add_seq(1)
    assert bm.append(1, 7).tolist() == [28, 29, 30, 31, 4, 5, 6]
    bm.fork(1, 2)
    assert bm.ref_count(7) == 2 and bm.ref_count(1) == 2
    assert bm.append(1, 1).tolist() == [15]
    assert bm.take_copies().tolist() == [[1, 3]]
    assert bm.block_table(1).tolist() == [7, 3] and bm.block_table(2).tolist() == [7, 1]
    assert (bm.ref_count(7), bm.ref_count(1), bm.ref_count(3)) == (2, 1, 1)
    assert bm.append(2, 1).tolist() == [7]
    assert bm.take_copies().shape == (0, 2)


@pytest.mark.parametrize("seed", range(25))
def test_random_sequences_match_oracle_bit_exactly(seed):
    rng = random.Random(1000 + seed)
    B = rng.choice([1, 2, 4, 16])
    N = rng.randint(3, 48)
    order = rng.sample(range(N), N)
    ref = BlockAllocator(N, B, order)
    bm = pa.BlockManager(N, B, order)
    live, nxt = [], 0
    for _ in range(250):
        op = rng.random()
        if op < 0.2 or not live:
            ref.add_seq(nxt)
            bm.add_seq(nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.65:
            s = rng.choice(live)
            n = rng.randint(0, 2 * B + 2)
            try:
                want = ref.append(s, n)
            except NoFreeBlocks:
                with pytest.raises(pa.PAError) as e:
                    bm.append(s, n)
                assert e.value.status == 5
            except TooLarge:
                with pytest.raises(pa.PAError) as e:
                    bm.append(s, n)
                assert e.value.status == 6
            else:
                assert bm.append(s, n).tolist() == want
            assert [list(p) for p in ref.take_copies()] == bm.take_copies().tolist()
        elif op < 0.8:
            p = rng.choice(live)
            ref.fork(p, nxt)
            bm.fork(p, nxt)
            live.append(nxt)
            nxt += 1
        else:
            s = live.pop(rng.randrange(len(live)))
            ref.free_seq(s)
            bm.free_seq(s)
        _compare(ref, bm, live)


@pytest.mark.parametrize("cfg,size", [(1, "full"), (2, "small"), (3, "small"), (4, "small"), (5, "small"),
                                      (3, "full"), (4, "full"), (5, "full")])
def test_workload_accounting_matches_oracle(cfg, size):
    wl = workloads.build(cfg, size)
    ref, slots, copies = run_allocator(wl)
    bm = pa.BlockManager(wl.num_blocks, wl.spec.block_size, wl.free_order)
    for ph, want_slots, want_copies in zip(wl.phases(), slots, copies):
        got = []
        for op in ph.ops:
            if op[0] == "add":
                bm.add_seq(op[1])
            elif op[0] == "fork":
                bm.fork(op[1], op[2])
            else:
                got.append(bm.append(op[1], op[2]))
        got = np.concatenate(got) if got else np.zeros(0, np.int64)
        assert np.array_equal(got, want_slots)
        assert bm.take_copies().tolist() == [list(p) for p in want_copies]
    seqs = [s for s, _ in wl.step.batch]
    width = max(len(ref.block_table(s)) for s in seqs)
    table, lens = bm.batch_tables(seqs, width)
    for i, s in enumerate(seqs):
        t = ref.block_table(s)
        assert table[i, : len(t)].tolist() == t and not table[i, len(t):].any()
        assert lens[i] == ref.seq_len(s)


def test_batched_append_matches_sequential_appends():
    rng = random.Random(7)
    order = rng.sample(range(64), 64)
    ref = BlockAllocator(64, 4, order)
    bm = pa.BlockManager(64, 4, order)
    for sq in range(6):
        ref.add_seq(sq)
        bm.add_seq(sq)
    ref.append(0, 5)
    bm.append(0, 5)
    ref.fork(0, 6)
    bm.fork(0, 6)
    seqs = [0, 6, 1, 2, 3, 6, 4, 5]
    counts = [3, 2, 0, 9, 1, 4, 7, 2]
    want = [sl for sq, c in zip(seqs, counts) for sl in ref.append(sq, c)]
    got = bm.append_batch(seqs, counts)
    assert got.tolist() == want
    assert [list(p) for p in ref.take_copies()] == bm.take_copies().tolist()
    _compare(ref, bm, range(7))


def test_batched_append_stops_at_first_failure():
    bm = pa.BlockManager(4, 4, range(4))
    for sq in range(3):
        bm.add_seq(sq)
    with pytest.raises(pa.PAError) as e:
        bm.append_batch([0, 1, 2], [8, 8, 1])  # the second needs 2 blocks, only 2 left -> ok; third fails
    assert e.value.status == 5 and "after 2 entries" in str(e.value)
    assert bm.seq_len(0) == 8 and bm.seq_len(1) == 8 and bm.seq_len(2) == 0


def test_end_to_end_loops_fit_the_tables_and_the_pool():
    """bench.py's end-to-end loops append one token to each of the GQA batch's 256 requests
    per step (two loops of warm-up, graph check and timed steps): the host block manager,
    replaying the workload's script, must still give every request a table within the
    tables' width and find free blocks for every append."""
    import bench

    wl = workloads.build(3)
    bm = pa.BlockManager(wl.num_blocks, wl.spec.block_size, wl.free_order)
    for ph in list(wl.setup) + [wl.step]:
        for op in ph.ops:
            assert op[0] in ("add", "append"), op[0]
            if op[0] == "add":
                bm.add_seq(op[1])
            else:
                bm.append(op[1], op[2])
        bm.take_copies()
    seqs = np.asarray([s for s, _ in wl.step.batch], np.int64)
    ones = np.ones(len(seqs), np.int64)
    slots = np.empty(len(seqs), np.int64)
    steps = 2 * (bench.E2E_STEPS + bench.E2E_WARMUP + 2)
    for _ in range(steps):
        bm.append_batch(seqs, ones, out=slots)
        table, lens = bm.batch_tables(seqs, bench.E2E_TABLE_WIDTH)
    assert int(lens.max()) <= bench.E2E_TABLE_WIDTH * wl.spec.block_size
    assert bm.num_free() >= 0
