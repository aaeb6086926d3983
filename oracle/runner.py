"""Run a seeded workload through the oracle: block manager, copies, writes, attention.

Test infrastructure (see the package docstring). Follows the phase rule stated
in ``workloads.configs``: operations, then the emitted copy pairs, then the
K/V writes, then the batch's attention.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .attention import BlockStore, copy_blocks_ref, kv_write_ref, paged_attention_ref, to_f64
from .block_manager import BlockAllocator
from .fp8 import dequantize, kv_write_fp8_ref
from .prefix_cache import PrefixCachingAllocator
from .swap import SwappingAllocator, SwappingPrefixAllocator


@dataclass
class OracleResult:
    allocator: BlockAllocator
    phase_slots: list = field(default_factory=list)  # per phase: int64 slot_mapping (op order)
    phase_copies: list = field(default_factory=list)  # per phase: list of (src, dst)
    k_cache: object = None
    v_cache: object = None
    block_table: np.ndarray = None  # int32 [S, max_blocks] (unused entries 0)
    seq_lens: np.ndarray = None  # int32 [S] after the step
    query_start_loc: np.ndarray = None  # int32 [S+1] of the step's batch
    batch_seqs: list = None  # the sequence of each batch entry
    q: np.ndarray = None  # [T, Hq, D] storage array of the step's queries
    out: np.ndarray = None  # float64 [T, Hq, D] (NaN rows for sequences not evaluated)


def run_script(wl):
    """Block-manager side only, every phase: (allocator, slots per phase, copy pairs per
    phase, appended ranges (seq, start, n) per phase in operation order)."""
    return run_script_swaps(wl)[:4]


def run_script_swaps(wl):
    """``run_script`` plus, per phase, the swaps in operation order: ("out" | "in", pairs)."""
    if wl.cpu_blocks:
        cls = SwappingPrefixAllocator if wl.prefix_caching else SwappingAllocator
        alloc = cls(wl.num_blocks, wl.spec.block_size, wl.free_order)
        alloc.enable_swap(wl.cpu_blocks, wl.cpu_free_order)
    elif wl.prefix_caching:
        alloc = PrefixCachingAllocator(wl.num_blocks, wl.spec.block_size, wl.free_order)
    else:
        alloc = BlockAllocator(wl.num_blocks, wl.spec.block_size, wl.free_order)

    def append(s, n):
        L = alloc.seq_len(s)
        if wl.prefix_caching:
            return alloc.append(s, n, tokens=wl.tokens(s, L, n).tolist())
        return alloc.append(s, n)

    slots_per_phase, copies_per_phase, appends_per_phase, swaps_per_phase = [], [], [], []
    for ph in wl.phases():
        slots, apps, swaps = [], [], []
        for op in ph.ops:
            if op[0] == "add":
                alloc.add_seq(op[1])
            elif op[0] == "fork":
                alloc.fork(op[1], op[2])
            elif op[0] == "append":
                apps.append((op[1], alloc.seq_len(op[1]), op[2]))
                slots.extend(append(op[1], op[2]))
            elif op[0] == "prompt":
                s, n = op[1], op[2]
                if wl.prefix_caching:  # reuse what the cache holds, compute the rest
                    hit = alloc.add_seq_cached(s, wl.tokens(s, 0, n).tolist(), max_hit=n - 1)
                else:
                    alloc.add_seq(s)
                    hit = 0
                apps.append((s, hit, n - hit))
                slots.extend(append(s, n - hit))
            elif op[0] == "fill":
                n = alloc.num_free() * wl.spec.block_size
                apps.append((op[1], 0, n))
                slots.extend(append(op[1], n))
            elif op[0] == "free":
                alloc.free_seq(op[1])
            elif op[0] == "swap_out":
                swaps.append(("out", alloc.swap_out(list(op[1]))))
            elif op[0] == "swap_in":
                swaps.append(("in", alloc.swap_in(list(op[1]))))
        slots_per_phase.append(np.asarray(slots, np.int64))
        copies_per_phase.append(alloc.take_copies())
        appends_per_phase.append(apps)
        swaps_per_phase.append(swaps)
    return alloc, slots_per_phase, copies_per_phase, appends_per_phase, swaps_per_phase


def run_allocator(wl):
    """Block-manager side only: slots and copy pairs of every phase, final tables."""
    alloc, slots, copies, _ = run_script(wl)
    return alloc, slots, copies


def step_ranges(wl, alloc, step_appends):
    """(seq, start, q_len) of the step's query rows, from the allocator's final lengths."""
    seqs = [s for s, _ in wl.step.batch or []]
    appended = {}
    for s, _, n in step_appends:
        appended[s] = appended.get(s, 0) + n
    return wl.step_queries({s: alloc.seq_len(s) for s in seqs}, appended)


def batch_metadata(wl, alloc, ranges=None):
    """block_table / seq_lens / query_start_loc of the step's batch (batch order);
    ``ranges`` = step_ranges(...) where q_len depends on the block manager."""
    batch = wl.step.batch or []
    seqs = [s for s, _ in batch]
    tables = [alloc.block_table(s) for s in seqs]
    width = max([len(t) for t in tables] + [1])
    bt = np.zeros((len(seqs), width), np.int32)
    for i, t in enumerate(tables):
        bt[i, : len(t)] = t
    seq_lens = np.asarray([alloc.seq_len(s) for s in seqs], np.int32)
    qsl = np.zeros(len(seqs) + 1, np.int32)
    qsl[1:] = np.cumsum([q for _, _, q in ranges] if ranges is not None else [q for _, q in batch])
    return bt, seq_lens, qsl, seqs


def _dequantized(cache, scale):
    """An E4M3 cache (codes) as float64 values: code value * scale, block by block."""
    if isinstance(cache, BlockStore):
        out = BlockStore(*cache.shape, np.float64)
        for b, blk in cache.items():
            out[b] = dequantize(blk, scale)
        return out
    return dequantize(cache, scale)


def run_workload(wl, eval_seqs=None) -> OracleResult:
    """Execute ``wl`` in the oracle.

    eval_seqs=None: dense caches, every request evaluated. Otherwise ``eval_seqs``
    are indices into the step's batch; only the blocks those requests (and the
    requests they were forked from) write are kept, and only their rows computed.
    """
    from workloads import relevant_seqs

    sp = wl.spec
    alloc, slots_pp, copies_pp, apps_pp, swaps_pp = run_script_swaps(wl)
    store_dtype = np.float32 if sp.dtype == "f32" else np.uint16
    fp8 = wl.kv_cache == "fp8_e4m3"
    cache_dtype = np.uint8 if fp8 else store_dtype  # E4M3 codes, or the inputs' storage type
    batch = wl.step.batch or []
    if eval_seqs is None:
        shape = (wl.num_blocks, sp.block_size, sp.num_kv_heads, sp.head_dim)
        kc, vc = np.zeros(shape, cache_dtype), np.zeros(shape, cache_dtype)
        relevant = None
    else:
        kc = BlockStore(sp.block_size, sp.num_kv_heads, sp.head_dim, cache_dtype)
        vc = BlockStore(sp.block_size, sp.num_kv_heads, sp.head_dim, cache_dtype)
        relevant = relevant_seqs(wl, [batch[i][0] for i in eval_seqs])
    ck = cv = None
    if wl.cpu_blocks:  # the CPU pool (always dense: it is small)
        cshape = (wl.cpu_blocks, sp.block_size, sp.num_kv_heads, sp.head_dim)
        ck, cv = np.zeros(cshape, cache_dtype), np.zeros(cshape, cache_dtype)
    for slots, copies, apps, swaps in zip(slots_pp, copies_pp, apps_pp, swaps_pp):
        copy_blocks_ref(kc, vc, copies)
        for direction, pairs in swaps:  # block copies between the pools, in operation order
            src, dst = ((kc, vc), (ck, cv)) if direction == "out" else ((ck, cv), (kc, vc))
            for s_blk, d_blk in pairs:
                for a_src, a_dst in zip(src, dst):
                    blk = a_src.get(s_blk) if isinstance(a_src, BlockStore) else a_src[s_blk]
                    if blk is None:
                        continue
                    if isinstance(a_dst, BlockStore):
                        a_dst[d_blk] = np.array(blk)
                    else:
                        a_dst[d_blk] = blk
        reqs = [a for a in apps if relevant is None or a[0] in relevant]
        vals = dict(zip(reqs, wl.kv_many(reqs))) if reqs else {}
        t0 = 0
        for a in apps:
            n = a[2]
            if a in vals:
                k, v = vals[a]
                if fp8:
                    kv_write_fp8_ref(kc, vc, to_f64(k).astype(np.float32), to_f64(v).astype(np.float32),
                                     slots[t0 : t0 + n], sp.block_size, wl.k_scale, wl.v_scale)
                else:
                    kv_write_ref(kc, vc, k, v, slots[t0 : t0 + n], sp.block_size)
            t0 += n
    ranges = step_ranges(wl, alloc, apps_pp[-1])
    bt, seq_lens, qsl, seqs = batch_metadata(wl, alloc, ranges)
    q = np.concatenate([wl.q(s, start, n) for s, start, n in ranges] or
                       [np.zeros((0, sp.num_heads, sp.head_dim), store_dtype)])
    ka, va = (_dequantized(kc, wl.k_scale), _dequantized(vc, wl.v_scale)) if fp8 else (kc, vc)
    out = paged_attention_ref(q, ka, va, bt, seq_lens, qsl, sp.scale, sp.block_size, seqs=eval_seqs)
    return OracleResult(alloc, slots_pp, copies_pp, kc, vc, bt, seq_lens, qsl, seqs, q, out)
