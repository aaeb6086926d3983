"""Oracle KV write, block copy and paged attention, in float64.

Test infrastructure (see the package docstring). Written for clarity: Python
loops over tokens and positions, NumPy only for the per-row dot products.

A cache is anything indexable by a physical block id that yields a [B, Hkv, D]
array: a NumPy array [num_blocks, B, Hkv, D] or a ``BlockStore`` (a dict of the
blocks actually written, used to evaluate a subset of a large batch). Caches
hold the storage type of the inputs: float32, or bfloat16 as uint16 bit patterns.

Sources:
- vLLM 0.10.0 flow page (ascendai.csdn.net), §3.3 KV Manager模块: slot =
  block * B + offset; the model runner hands ``slot_mapping`` to attention,
  which finds each token's K/V in the physical blocks. §3.5 Attention模块: q is
  the flattened token sequence of the batch, requests are told apart by
  ``query_start_loc``; K/V come from the whole cache through the block table.
- vLLM docs page (docs.acceleratez.fun, "vLLM"), PagedAttention › 算法流程
  step 2c/3d (store each token's KV in its physical block) and Copy-on-Write ›
  写时复制 (copy the old block's whole content into the new block).
- vLLM code-reading page (sourceaix.com), §5.1.1: attention is computed over
  the logical blocks, i.e. as if the tokens were contiguous.
- VLLM overview page (dn008.com.cn), §2.1 KV Cache 机制: decoder attention
  applies a causal mask after Q·Kᵀ so each token sees only earlier tokens.

Readings: the softmax scale multiplies the logits; query j of a request with
q_len queries and seq_len keys sits at position seq_len - q_len + j and sees
keys 0..that position; query head h reads KV head h // (Hq / Hkv); a negative
slot is padding and is skipped.
"""
from __future__ import annotations

import numpy as np


def to_f64(x: np.ndarray) -> np.ndarray:
    """Storage array -> float64. uint16 holds bfloat16: the upper half of a binary32."""
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


class BlockStore(dict):
    """A sparse cache: block id -> [B, Hkv, D] array, created on first write."""

    def __init__(self, block_size, num_kv_heads, head_dim, dtype):
        super().__init__()
        self.shape = (block_size, num_kv_heads, head_dim)
        self.dtype = dtype

    def block_for_write(self, b):
        if b not in self:
            self[b] = np.zeros(self.shape, self.dtype)
        return self[b]


def _block_for_write(cache, b):
    return cache.block_for_write(b) if isinstance(cache, BlockStore) else cache[b]


def kv_write_ref(k_cache, v_cache, k, v, slot_mapping, block_size, keep=None):
    """cache[slot // B, slot % B] = token's K (and V) for every slot >= 0.

    ``keep`` (optional set of token indices) restricts the write to those tokens.
    """
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0 or (keep is not None and t not in keep):
            continue
        b, off = slot // block_size, slot % block_size
        _block_for_write(k_cache, b)[off] = k[t]
        _block_for_write(v_cache, b)[off] = v[t]


def copy_blocks_ref(k_cache, v_cache, pairs):
    """For each (src, dst) in order: the whole block dst becomes a copy of src."""
    for src, dst in pairs:
        src, dst = int(src), int(dst)
        if isinstance(k_cache, BlockStore):
            if src not in k_cache:
                continue  # a block no evaluated sequence reads
            k_cache[dst] = k_cache[src].copy()
            v_cache[dst] = v_cache[src].copy()
        else:
            k_cache[dst] = k_cache[src]
            v_cache[dst] = v_cache[src]


def gather_kv(cache, table, seq_len, block_size):
    """Logical K (or V) of one request, [seq_len, Hkv, D] float64, read position by position."""
    rows = []
    for p in range(seq_len):
        rows.append(cache[int(table[p // block_size])][p % block_size])
    return to_f64(np.stack(rows))


def attend(q, K, V, scale, q_positions):
    """Causal softmax attention of query rows against contiguous keys.

    q: [n, Hq, D]; K, V: [L, Hkv, D] (float64); q_positions[j] = the position of
    query row j, which sees keys 0..q_positions[j]. Returns [n, Hq, D] float64.
    """
    n, Hq, D = q.shape
    Hkv = K.shape[1]
    group = Hq // Hkv
    out = np.zeros((n, Hq, D))
    for j in range(n):
        last = int(q_positions[j])
        for h in range(Hq):
            g = h // group
            keys = K[: last + 1, g, :]
            logits = scale * (keys @ q[j, h])
            w = np.exp(logits - logits.max())
            w /= w.sum()
            out[j, h] = w @ V[: last + 1, g, :]
    return out


def paged_attention_ref(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, scale, block_size,
                        seqs=None):
    """Attention of every request of a batch through its block table.

    q: [T, Hq, D] storage array (T = query_start_loc[-1]); block_table[s] lists
    request s's physical blocks in logical order. Returns float64 [T, Hq, D];
    with ``seqs`` given, only those requests' rows are computed (others are NaN).
    """
    T = int(query_start_loc[-1])
    out = np.full((T,) + q.shape[1:], np.nan)
    qf = to_f64(q)
    S = len(seq_lens)
    for s in range(S) if seqs is None else seqs:
        a, b = int(query_start_loc[s]), int(query_start_loc[s + 1])
        q_len, L = b - a, int(seq_lens[s])
        if q_len == 0:
            continue
        K = gather_kv(k_cache, block_table[s], L, block_size)
        V = gather_kv(v_cache, block_table[s], L, block_size)
        out[a:b] = attend(qf[a:b], K, V, scale, [L - q_len + j for j in range(q_len)])
    return out


def dense_causal_ref(q, k, v, scale):
    """The same attention over contiguous K/V [L, Hkv, D] (no paging); q: [n, Hq, D]
    are the last n positions."""
    qf, K, V = to_f64(q), to_f64(k), to_f64(v)
    L, n = K.shape[0], qf.shape[0]
    return attend(qf, K, V, scale, [L - n + j for j in range(n)])
