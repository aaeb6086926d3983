"""Run a seeded workload through the oracle: block manager, copies, writes, attention.

Test infrastructure (see the package docstring). Follows the phase rule stated
in ``workloads.configs``: operations, then the emitted copy pairs, then the
K/V writes, then the batch's attention.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .attention import BlockStore, copy_blocks_ref, kv_write_ref, paged_attention_ref
from .block_manager import BlockAllocator


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


def run_allocator(wl):
    """Block-manager side only: slots and copy pairs of every phase, final tables."""
    alloc = BlockAllocator(wl.num_blocks, wl.spec.block_size, wl.free_order)
    slots_per_phase, copies_per_phase = [], []
    for ph in wl.phases():
        slots = []
        for op in ph.ops:
            if op[0] == "add":
                alloc.add_seq(op[1])
            elif op[0] == "fork":
                alloc.fork(op[1], op[2])
            elif op[0] == "append":
                slots.extend(alloc.append(op[1], op[2]))
        slots_per_phase.append(np.asarray(slots, np.int64))
        copies_per_phase.append(alloc.take_copies())
    return alloc, slots_per_phase, copies_per_phase


def batch_metadata(wl, alloc):
    """block_table / seq_lens / query_start_loc of the step's batch (batch order)."""
    batch = wl.step.batch or []
    seqs = [s for s, _ in batch]
    tables = [alloc.block_table(s) for s in seqs]
    width = max([len(t) for t in tables] + [1])
    bt = np.zeros((len(seqs), width), np.int32)
    for i, t in enumerate(tables):
        bt[i, : len(t)] = t
    seq_lens = np.asarray([alloc.seq_len(s) for s in seqs], np.int32)
    qsl = np.zeros(len(seqs) + 1, np.int32)
    qsl[1:] = np.cumsum([q for _, q in batch])
    return bt, seq_lens, qsl, seqs


def run_workload(wl, eval_seqs=None) -> OracleResult:
    """Execute ``wl`` in the oracle.

    eval_seqs=None: dense caches, every request evaluated. Otherwise ``eval_seqs``
    are indices into the step's batch; only the blocks those requests (and the
    requests they were forked from) write are kept, and only their rows computed.
    """
    from workloads import relevant_seqs

    sp = wl.spec
    alloc, slots_pp, copies_pp = run_allocator(wl)
    store_dtype = np.float32 if sp.dtype == "f32" else np.uint16
    batch = wl.step.batch or []
    if eval_seqs is None:
        shape = (wl.num_blocks, sp.block_size, sp.num_kv_heads, sp.head_dim)
        kc, vc = np.zeros(shape, store_dtype), np.zeros(shape, store_dtype)
        relevant = None
    else:
        kc = BlockStore(sp.block_size, sp.num_kv_heads, sp.head_dim, store_dtype)
        vc = BlockStore(sp.block_size, sp.num_kv_heads, sp.head_dim, store_dtype)
        relevant = relevant_seqs(wl, [batch[i][0] for i in eval_seqs])
    lens = {}
    for ph, slots, copies in zip(wl.phases(), slots_pp, copies_pp):
        apps = wl.appends(ph, lens)
        copy_blocks_ref(kc, vc, copies)
        reqs = [a for a in apps if relevant is None or a[0] in relevant]
        vals = dict(zip(reqs, wl.kv_many(reqs))) if reqs else {}
        t0 = 0
        for a in apps:
            n = a[2]
            if a in vals:
                k, v = vals[a]
                kv_write_ref(kc, vc, k, v, slots[t0 : t0 + n], sp.block_size)
            t0 += n
    bt, seq_lens, qsl, seqs = batch_metadata(wl, alloc)
    q = np.concatenate([wl.q(s, start, n) for s, start, n in wl.step_queries()] or
                       [np.zeros((0, sp.num_heads, sp.head_dim), store_dtype)])
    out = paged_attention_ref(q, kc, vc, bt, seq_lens, qsl, sp.scale, sp.block_size, seqs=eval_seqs)
    return OracleResult(alloc, slots_pp, copies_pp, kc, vc, bt, seq_lens, qsl, seqs, q, out)
