"""The C++ block manager's swapping against the oracle, bit for bit (CPU only).

Seeded random scripts of admissions, appends, forks, releases and group swaps (with and
without prefix caching) on pools small enough to run out: after every operation both sides
agree on statuses, copy pairs (copy-on-write and swap), tables, lengths, both pools'
reference counts and free queues.
"""
import random

import numpy as np
import pytest

import paged_kv_cache_161_gb300 as pa
from oracle import NoFreeBlocks, TooLarge
from oracle.swap import SwappingAllocator, SwappingPrefixAllocator


def _run(fn):
    try:
        return 0, fn()
    except pa.PAError as e:
        return e.status, None
    except NoFreeBlocks:
        return 5, None
    except TooLarge:
        return 6, None
    except ValueError:
        return 1, None


@pytest.mark.parametrize("prefix", [False, True])
@pytest.mark.parametrize("seed", range(12))
def test_random_swap_scripts_match_oracle(seed, prefix):
    rng = random.Random(500 + seed)
    B = rng.choice([1, 2, 4, 8, 16])
    NB, NC = rng.randint(6, 40), rng.randint(3, 40)
    order, corder = list(range(NB)), list(range(NC))
    rng.shuffle(order)
    rng.shuffle(corder)
    c = pa.BlockManager(NB, B, order)
    if prefix:
        c.enable_prefix_caching()
    c.enable_swap(NC, corder)
    o = (SwappingPrefixAllocator if prefix else SwappingAllocator)(NB, B, order)
    o.enable_swap(NC, corder)
    live, nxt, swaps = [], 0, 0
    for _ in range(250):
        op = rng.random()
        if op < 0.2 or not live:
            toks = [rng.randrange(3) for _ in range(rng.randint(1, 3 * B))]
            s, nxt = nxt, nxt + 1
            if prefix:
                hc = c.add_seq_cached(s, toks, len(toks) - 1)
                ho = o.add_seq_cached(s, toks, max_hit=len(toks) - 1)
                assert hc == ho
                r_c = _run(lambda: c.append_tokens(s, toks[hc:]))
                r_o = _run(lambda: o.append(s, len(toks) - ho, tokens=toks[ho:]))
            else:
                c.add_seq(s)
                o.add_seq(s)
                r_c = _run(lambda: c.append(s, len(toks)))
                r_o = _run(lambda: o.append(s, len(toks)))
            live.append(s)
        elif op < 0.45:
            s = rng.choice(live)
            toks = [rng.randrange(3) for _ in range(rng.randint(1, B + 1))]
            if prefix:
                r_c = _run(lambda: c.append_tokens(s, toks))
                r_o = _run(lambda: o.append(s, len(toks), tokens=toks))
            else:
                r_c = _run(lambda: c.append(s, len(toks)))
                r_o = _run(lambda: o.append(s, len(toks)))
        elif op < 0.55:
            p = rng.choice(live)
            r_c = _run(lambda: c.fork(p, nxt))
            r_o = _run(lambda: o.fork(p, nxt))
            if r_c[0] == 0:
                live.append(nxt)
            nxt += 1
        elif op < 0.8:
            group = rng.sample(live, rng.randint(1, min(3, len(live))))
            if rng.random() < 0.5:
                r_c = _run(lambda: c.swap_out(group))
                r_o = _run(lambda: o.swap_out(group))
            else:
                r_c = _run(lambda: c.swap_in(group))
                r_o = _run(lambda: o.swap_in(group))
            swaps += r_c[0] == 0
        else:
            s = rng.choice(live)
            c.free_seq(s)
            o.free_seq(s)
            live.remove(s)
            r_c = r_o = (0, None)
        assert r_c[0] == r_o[0], (r_c, r_o)
        if r_c[0] == 0 and r_c[1] is not None:
            assert np.asarray(r_c[1]).tolist() == [list(p) if isinstance(p, tuple) else p for p in r_o[1]]
        assert c.take_copies().tolist() == [list(p) for p in o.take_copies()]
        assert c.free_queue().tolist() == list(o.free)
        assert c.num_free_cpu() == len(o.cpu_free)
        for s in live:
            assert c.block_table(s).tolist() == o.block_table(s)
            assert c.seq_len(s) == o.seq_len(s)
            assert c.is_swapped(s) == (s in o.swapped)
        for b in range(NB):
            assert c.ref_count(b) == o.ref_count(b)
        for b in range(NC):
            assert c.cpu_ref_count(b) == o.cpu_ref[b]
    assert swaps > 0


def test_swap_argument_rules():
    m = pa.BlockManager(8, 4, list(range(8)))
    with pytest.raises(pa.PAError):
        m.swap_out([0])  # swapping not enabled
    m.enable_swap(4, [3, 2, 1, 0])
    m.add_seq(0)
    m.append(0, 6)
    with pytest.raises(pa.PAError):
        m.swap_in([0])  # not swapped
    with pytest.raises(pa.PAError):
        m.swap_out([0, 0])  # repeated
    pairs = m.swap_out([0])
    assert pairs.tolist() == [[0, 3], [1, 2]] and m.is_swapped(0)
    with pytest.raises(pa.PAError):
        m.append(0, 1)  # frozen while swapped
    with pytest.raises(pa.PAError):
        m.batch_tables([0], 4)  # its blocks are not on the GPU
    m.free_seq(0)
    assert m.num_free_cpu() == 4 and m.num_free() == 8
