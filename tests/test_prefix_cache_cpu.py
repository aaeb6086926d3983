"""The C++ block manager's prefix caching against the oracle, bit for bit (CPU only).

After every operation of seeded random scripts (admissions that look up the cache,
appends with token ids, forks, releases, on pools small enough to evict), both sides
must agree on reused-token counts, slots, copy pairs, block tables, lengths, reference
counts, the free list order, the number of registered blocks and evictions.
"""
import random

import numpy as np
import pytest

import paged_kv_cache_161_gb300 as pa
from oracle import NoFreeBlocks, PrefixCachingAllocator, TooLarge


def _same_state(c, o, live):
    assert c.free_queue().tolist() == list(o.free)
    for s in live:
        assert c.block_table(s).tolist() == o.block_table(s)
        assert c.seq_len(s) == o.seq_len(s)
    for b in range(o.num_blocks):
        assert c.ref_count(b) == o.ref_count(b)
    cached, hit_blocks, evictions = c.prefix_stats()
    assert cached == o.num_cached() and hit_blocks == o.hits and evictions == o.evictions


def _status(fn):
    try:
        return 0, fn()
    except pa.PAError as e:
        return e.status, None
    except NoFreeBlocks:
        return 5, None
    except TooLarge:
        return 6, None


@pytest.mark.parametrize("seed", range(16))
def test_random_scripts_match_oracle(seed):
    rng = random.Random(1000 + seed)
    B = rng.choice([1, 2, 4, 8, 16])
    NB = rng.randint(6, 48)
    order = list(range(NB))
    rng.shuffle(order)
    c = pa.BlockManager(NB, B, order)
    c.enable_prefix_caching()
    o = PrefixCachingAllocator(NB, B, order)
    vocab = rng.choice([2, 3, 50])
    bases = [[rng.randrange(vocab) for _ in range(rng.randint(0, 5 * B))] for _ in range(4)]
    live, nxt = [], 0
    for _ in range(250):
        op = rng.random()
        if op < 0.3 or not live:
            prompt = list(rng.choice(bases)) + [rng.randrange(vocab) for _ in range(rng.randint(1, 2 * B))]
            s, nxt = nxt, nxt + 1
            hc = c.add_seq_cached(s, prompt, max_hit=len(prompt) - 1)
            ho = o.add_seq_cached(s, prompt, max_hit=len(prompt) - 1)
            assert hc == ho
            live.append(s)
            st_c, sl_c = _status(lambda: c.append_tokens(s, prompt[hc:]))
            st_o, sl_o = _status(lambda: o.append(s, len(prompt) - ho, tokens=prompt[ho:]))
        elif op < 0.6:
            s = rng.choice(live)
            toks = [rng.randrange(vocab) for _ in range(rng.randint(1, 2 * B))]
            st_c, sl_c = _status(lambda: c.append_tokens(s, toks))
            st_o, sl_o = _status(lambda: o.append(s, len(toks), tokens=toks))
        elif op < 0.75:
            p = rng.choice(live)
            c.fork(p, nxt)
            o.fork(p, nxt)
            live.append(nxt)
            nxt += 1
            st_c = st_o = 0
            sl_c = sl_o = []
        else:
            s = rng.choice(live)
            c.free_seq(s)
            o.free_seq(s)
            live.remove(s)
            st_c = st_o = 0
            sl_c = sl_o = []
        assert st_c == st_o
        if st_c == 0:
            assert list(np.asarray(sl_c).tolist()) == list(sl_o)
        assert c.take_copies().tolist() == [list(p) for p in o.take_copies()]
        _same_state(c, o, live)


def test_batched_token_append_matches_single_appends():
    B, NB = 4, 64
    a = pa.BlockManager(NB, B, list(range(NB)))
    b = pa.BlockManager(NB, B, list(range(NB)))
    for m in (a, b):
        m.enable_prefix_caching()
    rng = np.random.default_rng(3)
    seqs = [0, 1, 2]
    prompts = [rng.integers(0, 5, size=n).tolist() for n in (9, 13, 4)]
    for s, p in zip(seqs, prompts):
        assert a.add_seq_cached(s, p, len(p) - 1) == b.add_seq_cached(s, p, len(p) - 1) == 0
    counts = [len(p) for p in prompts]
    flat = [t for p in prompts for t in p]
    got = a.append_tokens_batch(seqs, counts, flat)
    want = np.concatenate([b.append_tokens(s, p) for s, p in zip(seqs, prompts)])
    assert got.tolist() == want.tolist()
    assert a.prefix_stats() == b.prefix_stats()


def test_prefix_caching_argument_rules():
    m = pa.BlockManager(8, 4, list(range(8)))
    m.add_seq(0)
    with pytest.raises(pa.PAError):
        m.enable_prefix_caching()  # only on a fresh manager
    with pytest.raises(pa.PAError):
        m.add_seq_cached(1, [1, 2, 3, 4, 5], 4)  # caching not enabled
    m2 = pa.BlockManager(8, 4, list(range(8)))
    m2.enable_prefix_caching()
    m2.add_seq(0)
    with pytest.raises(pa.PAError):
        m2.append(0, 3)  # token ids are required once caching is on
    assert m2.append_tokens(0, [7, 8, 9]).tolist() == [0, 1, 2]
    with pytest.raises(pa.PAError):
        m2.add_seq_cached(0, [1, 2], 1)  # id in use


@pytest.mark.parametrize("size", ["small", "full"])
@pytest.mark.parametrize("caching", [True, False])
def test_system_prompt_script_matches_oracle(size, caching):
    """The system-prompt workload's script on the C++ manager: same reused counts, slots,
    copy pairs and tables as the oracle; with caching every request reuses all of the
    system prompt's full blocks."""
    import workloads
    from oracle import run_script

    wl = workloads.system_prompt(size, caching=caching)
    alloc, slots_pp, copies_pp, apps_pp = run_script(wl)
    bm = pa.BlockManager(wl.num_blocks, wl.spec.block_size, wl.free_order)
    if caching:
        bm.enable_prefix_caching()
    for ph, want_slots, want_copies, want_apps in zip(wl.phases(), slots_pp, copies_pp, apps_pp):
        got, apps = [], []
        for op in ph.ops:
            if op[0] == "prompt":
                s, n = op[1], op[2]
                hit = bm.add_seq_cached(s, wl.tokens(s, 0, n), n - 1) if caching else (bm.add_seq(s) or 0)
                apps.append((s, hit, n - hit))
                got.append(bm.append_tokens(s, wl.tokens(s, hit, n - hit)) if caching else bm.append(s, n))
            elif op[0] == "free":
                bm.free_seq(op[1])
        assert apps == want_apps
        assert np.array_equal(np.concatenate(got) if got else np.zeros(0, np.int64), want_slots)
        assert bm.take_copies().tolist() == [list(p) for p in want_copies]
    B, P = wl.spec.block_size, wl.meta["system_len"]
    for s, hit, _ in apps_pp[-1]:
        assert hit == ((P // B) * B if caching else 0)
        assert bm.block_table(s).tolist() == alloc.block_table(s)
    if caching:
        cached, hits, evictions = bm.prefix_stats()
        assert hits == wl.meta["requests"] * (P // B) and evictions == 0


def test_batch_groups_from_shared_tables():
    """pa_bm_batch_groups on the shared-prefix workload: each prompt's samples form a group
    whose shared length is the longest run of identical leading blocks (brute force over
    the oracle's tables), capped by the shortest member."""
    import workloads
    from oracle import run_allocator

    wl = workloads.build(4, "small")
    ref, _, _ = run_allocator(wl)
    bm = pa.BlockManager(wl.num_blocks, wl.spec.block_size, wl.free_order)
    for ph in wl.phases():
        for op in ph.ops:
            if op[0] == "add":
                bm.add_seq(op[1])
            elif op[0] == "fork":
                bm.fork(op[1], op[2])
            else:
                bm.append(op[1], op[2])
        bm.take_copies()
    seqs = [s for s, _ in wl.step.batch]
    sg, gr, sl = bm.batch_groups(seqs, max_members=4)
    n_samp = wl.meta["samples"]
    assert len(gr) == wl.meta["prompts"]
    B = wl.spec.block_size
    for g, (a, b) in enumerate(gr.tolist()):
        assert b - a == n_samp and all(sg[a:b] == g)
        tabs = [ref.block_table(seqs[i]) for i in range(a, b)]
        k = 0
        while all(len(t) > k for t in tabs) and len({t[k] for t in tabs}) == 1:
            k += 1
        assert sl[g] == min(k * B, min(ref.seq_len(seqs[i]) for i in range(a, b)))
    sg2, gr2, _ = bm.batch_groups(seqs, max_members=2)
    assert len(gr2) == 2 * wl.meta["prompts"] and (gr2[:, 1] - gr2[:, 0] == 2).all()
