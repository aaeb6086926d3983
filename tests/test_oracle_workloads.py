"""The oracle run end to end on the seeded workloads (CPU only).

Reading every request's tokens back through its final block table must give
exactly the K/V stream that was appended to it (or to the request it was forked
from), and attention over the paged cache must equal brute-force attention over
that contiguous stream.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import dense_causal_ref, run_allocator, run_workload, to_f64


def _streams(wl, seq):
    """The logical K/V stream of ``seq`` rebuilt from the workload's append script."""
    parts, lens, parent = {}, {}, {}
    for ph in wl.phases():
        for op in ph.ops:
            if op[0] == "add":
                parts[op[1]], lens[op[1]] = [], 0
            elif op[0] == "fork":
                parts[op[2]] = list(parts[op[1]])
                lens[op[2]] = lens[op[1]]
            elif op[0] == "append":
                parts[op[1]].append(wl.kv(op[1], lens[op[1]], op[2]))
                lens[op[1]] += op[2]
    ks = np.concatenate([p[0] for p in parts[seq]])
    vs = np.concatenate([p[1] for p in parts[seq]])
    return ks, vs


def test_bf16_storage_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    ours = workloads.configs._to_storage(x, "bf16")
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def test_config1_tables_slots_and_positions():
    wl = workloads.build(1)
    alloc, slots, copies = run_allocator(wl)
    assert [alloc.seq_len(s) for s in range(3)] == [8, 17, 34]
    assert [len(alloc.block_table(s)) for s in range(3)] == [2, 5, 9]
    step = slots[-1]
    t = [alloc.block_table(s) for s in range(3)]
    # 7 -> 8 fills the last slot; 16 -> 17 opens a block; 33 -> 34 is mid-block
    assert step.tolist() == [t[0][1] * 4 + 3, t[1][4] * 4 + 0, t[2][8] * 4 + 1]
    assert all(c == [] for c in copies)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_small_workloads_read_back_and_match_dense(cfg):
    wl = workloads.build(cfg, "small")
    res = run_workload(wl)
    B = wl.spec.block_size
    for i, s in enumerate(res.batch_seqs):
        L = int(res.seq_lens[i])
        ks, vs = _streams(wl, s)
        assert len(ks) == L
        table = res.block_table[i]
        got_k = np.stack([res.k_cache[table[p // B]][p % B] for p in range(L)])
        got_v = np.stack([res.v_cache[table[p // B]][p % B] for p in range(L)])
        assert np.array_equal(got_k, ks) and np.array_equal(got_v, vs)
        a, b = res.query_start_loc[i], res.query_start_loc[i + 1]
        if b > a:
            want = dense_causal_ref(res.q[a:b], ks, vs, wl.spec.scale)
            assert np.max(np.abs(res.out[a:b] - want)) < 1e-12


def test_shared_prefix_accounting():
    wl = workloads.build(4, "small")
    alloc, slots, copies = run_allocator(wl)
    P, n, plen = wl.meta["prompts"], wl.meta["samples"], wl.meta["prompt_len"]
    B = wl.spec.block_size
    all_pairs = [p for c in copies for p in c]
    assert len(all_pairs) == P * (n - 1)  # every sharer but the last holder copies
    for p in range(P):
        tabs = [alloc.block_table(p * n + i) for i in range(n)]
        shared = plen // B
        for b in tabs[0][:shared]:
            assert alloc.ref_count(b) == n
            assert all(t[:shared] == tabs[0][:shared] for t in tabs)
        lasts = {t[shared] for t in tabs}
        assert len(lasts) == n  # the partial prompt block diverged into n private blocks
        assert all(alloc.ref_count(b) == 1 for b in lasts)


def test_sparse_evaluation_equals_dense():
    wl = workloads.build(4, "small")
    dense = run_workload(wl)
    pick = [1, 6, 11]
    sparse = run_workload(wl, eval_seqs=pick)
    for i in pick:
        a, b = dense.query_start_loc[i], dense.query_start_loc[i + 1]
        assert np.array_equal(dense.out[a:b], sparse.out[a:b])
    others = [i for i in range(len(dense.batch_seqs)) if i not in pick]
    assert np.isnan(sparse.out[[dense.query_start_loc[i] for i in others]]).all()


def test_mixed_batch_positions():
    wl = workloads.build(5, "small")
    res = run_workload(wl)
    C, chunk = wl.meta["chunks"], wl.meta["chunk_len"]
    qlens = np.diff(res.query_start_loc)
    assert qlens[:C].tolist() == [chunk] * C and (qlens[C:] == 1).all()
    assert res.seq_lens[:C].tolist() == [int(p) + chunk for p in wl.meta["prior"]]
    # first query of a chunk with no prior context sees only itself: out = its own V
    ks, vs = _streams(wl, 0)
    if wl.meta["prior"][0] == 0:
        G = wl.spec.num_heads // wl.spec.num_kv_heads
        assert np.allclose(res.out[0], np.repeat(to_f64(vs[0]), G, axis=0))


def test_full_size_shapes():
    for cfg, S in [(2, 64), (3, 256), (4, 256), (5, 256)]:
        wl = workloads.build(cfg)
        assert wl.num_seqs == S and len(wl.step.batch) == S
    wl3 = workloads.build(3)
    L = np.array(wl3.meta["final_lens"]) - 1
    assert L.min() >= 16 and L.max() <= 8192
    assert 700 < np.median(L) < 1400


def test_system_prompt_cached_rows_equal_uncached_rows():
    """With prefix caching a request computes only the rows after the reused prefix; those
    rows see the same keys and values and must equal the uncached run's rows exactly, and
    both must equal brute-force attention over the contiguous stream."""
    c = run_workload(workloads.system_prompt("small", caching=True))
    u = run_workload(workloads.system_prompt("small", caching=False))
    wl = workloads.system_prompt("small", caching=True)
    B, P = wl.spec.block_size, wl.meta["system_len"]
    hit = (P // B) * B
    for i, s in enumerate(c.batch_seqs):
        L = int(c.seq_lens[i])
        assert L == int(u.seq_lens[i]) == P + wl.meta["user_lens"][i]
        ca, cb = c.query_start_loc[i], c.query_start_loc[i + 1]
        ua, ub = u.query_start_loc[i], u.query_start_loc[i + 1]
        assert cb - ca == L - hit and ub - ua == L
        assert np.array_equal(c.out[ca:cb], u.out[ua + hit:ub])
        # the cached request's K/V stream: the warm request's prompt, then its own tokens
        ks, vs = wl.kv(s, 0, L)
        table = c.block_table[i]
        got_k = np.stack([c.k_cache[table[p // B]][p % B] for p in range(L)])
        assert np.array_equal(got_k, ks)
        want = dense_causal_ref(u.q[ua:ub], ks, vs, wl.spec.scale)
        assert np.max(np.abs(u.out[ua:ub] - want)) < 1e-12


@pytest.mark.parametrize("cfg", [3, 4, 5])
def test_fp8_workloads_read_back_and_match_dense(cfg):
    """Over an E4M3 cache every request reads back E4M3(x / scale) of its own K/V stream,
    and attention equals brute force over the dequantised stream."""
    from oracle import dequantize, quantize

    wl = workloads.with_fp8_cache(workloads.build(cfg, "small"), k_scale=2.0 ** -6, v_scale=0.0123)
    res = run_workload(wl)
    B = wl.spec.block_size
    for i, s in enumerate(res.batch_seqs):
        L = int(res.seq_lens[i])
        ks, vs = _streams(wl, s)
        table = res.block_table[i]
        got_k = np.stack([res.k_cache[table[p // B]][p % B] for p in range(L)])
        got_v = np.stack([res.v_cache[table[p // B]][p % B] for p in range(L)])
        assert np.array_equal(got_k, quantize(to_f64(ks).astype(np.float32), wl.k_scale))
        assert np.array_equal(got_v, quantize(to_f64(vs).astype(np.float32), wl.v_scale))
        a, b = res.query_start_loc[i], res.query_start_loc[i + 1]
        if b > a:
            want = dense_causal_ref(res.q[a:b], dequantize(got_k, wl.k_scale), dequantize(got_v, wl.v_scale),
                                    wl.spec.scale)
            assert np.max(np.abs(res.out[a:b] - want)) < 1e-12


def test_preemption_workload_reads_back_after_swapping():
    """The swapped-out group comes back (in other GPU blocks, after a long request
    overwrote its old ones) reading exactly its own streams; attention matches brute force."""
    from oracle import run_script_swaps

    wl = workloads.preemption("small")
    alloc, _, _, _, swaps = run_script_swaps(wl)
    out_pairs = [p for ph in swaps for d, pairs in ph if d == "out" for p in pairs]
    in_pairs = [p for ph in swaps for d, pairs in ph if d == "in" for p in pairs]
    assert len(out_pairs) == len(in_pairs) > 0
    res = run_workload(wl)
    B = wl.spec.block_size
    old_gpu = {g for g, _ in out_pairs}
    new_gpu = {g for _, g in in_pairs}
    assert old_gpu != new_gpu  # the group came back into other blocks
    for i, s in enumerate(res.batch_seqs):
        L = int(res.seq_lens[i])
        ks, vs = _streams(wl, s)
        table = res.block_table[i]
        got_k = np.stack([res.k_cache[table[p // B]][p % B] for p in range(L)])
        assert np.array_equal(got_k, ks)
        a, b = res.query_start_loc[i], res.query_start_loc[i + 1]
        want = dense_causal_ref(res.q[a:b], ks, vs, wl.spec.scale)
        assert np.max(np.abs(res.out[a:b] - want)) < 1e-12
