"""Pins of the oracle's writes, copies and attention (CPU only).

Each pin fixes the oracle against something other than itself: the bfloat16
definition, closed forms of the byte moves, a library attention routine
(torch's scaled_dot_product_attention in float64), brute force, invariances and
special cases of softmax attention.
"""
import numpy as np
import pytest
import torch

from oracle import (
    BlockStore,
    copy_blocks_ref,
    dense_causal_ref,
    kv_write_ref,
    paged_attention_ref,
    to_f64,
)


def test_bf16_decoding_matches_definition():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0001, 0x7F7F, 0x8000], np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0**-7, 2.0**-133, (2 - 2.0**-7) * 2.0**127, -0.0]
    got = to_f64(bits)
    assert got.tolist() == want
    assert np.signbit(got[-1])
    # and the same as torch's bfloat16 for random patterns (library cross-check)
    r = np.random.default_rng(0).integers(0, 0x7F80, 1000, dtype=np.uint16)
    t = torch.from_numpy(r.astype(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(to_f64(r), t)


def _sdpa(q, k, v, scale, q_pos):
    """torch SDPA in float64 with an explicit boolean mask and repeated KV heads."""
    n, Hq, D = q.shape
    L, Hkv, _ = k.shape
    G = Hq // Hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    mask = torch.arange(L)[None, :] <= torch.tensor(q_pos)[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("seed", range(8))
def test_dense_reference_equals_library_attention(seed):
    rng = np.random.default_rng(seed)
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4]))
    D = int(rng.choice([8, 16, 64]))
    L = int(rng.integers(1, 40))
    n = int(rng.integers(1, L + 1))
    scale = float(rng.uniform(0.05, 0.5))
    q = rng.standard_normal((n, Hq := Hkv * G, D))
    k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D))
    got = dense_causal_ref(q, k, v, scale)
    want = _sdpa(q, k, v, scale, [L - n + j for j in range(n)])
    assert np.max(np.abs(got - want)) < 1e-12
    assert Hq == q.shape[1]


def _paged_from_dense(rng, ks, vs, B, NB):
    """Write contiguous per-request K/V into a cache at random physical blocks."""
    Hkv, D = ks[0].shape[1:]
    kc = np.zeros((NB, B, Hkv, D))
    vc = np.zeros((NB, B, Hkv, D))
    perm = list(rng.permutation(NB))
    tables = []
    for k, v in zip(ks, vs):
        nblk = -(-len(k) // B)
        tab = [perm.pop() for _ in range(nblk)]
        tables.append(tab)
        slots = [tab[p // B] * B + p % B for p in range(len(k))]
        kv_write_ref(kc, vc, k, v, slots, B)
    width = max(len(t) for t in tables)
    bt = np.zeros((len(tables), width), np.int32)
    for i, t in enumerate(tables):
        bt[i, : len(t)] = t
    return kc, vc, bt


@pytest.mark.parametrize("seed", range(6))
def test_paged_equals_dense_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    B, Hkv, G, D = int(rng.choice([1, 4, 16])), 2, 2, 16
    lens = [int(x) for x in rng.integers(1, 40, size=4)]
    qlens = [int(rng.integers(1, L + 1)) if i % 2 else 1 for i, L in enumerate(lens)]
    ks = [rng.standard_normal((L, Hkv, D)) for L in lens]
    vs = [rng.standard_normal((L, Hkv, D)) for L in lens]
    qs = [rng.standard_normal((n, Hkv * G, D)) for n in qlens]
    kc, vc, bt = _paged_from_dense(rng, ks, vs, B, NB=sum(-(-L // B) for L in lens) + 5)
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    out = paged_attention_ref(np.concatenate(qs), kc, vc, bt, np.array(lens, np.int32), qsl, 0.25, B)
    for s in range(len(lens)):
        want = _sdpa(qs[s], ks[s], vs[s], 0.25, [lens[s] - qlens[s] + j for j in range(qlens[s])])
        assert np.max(np.abs(out[qsl[s]:qsl[s + 1]] - want)) < 1e-12


def test_output_invariant_under_physical_block_relabelling():
    rng = np.random.default_rng(7)
    B, NB, Hkv, D = 4, 32, 2, 8
    lens = [13, 5, 21]
    ks = [rng.standard_normal((L, Hkv, D)) for L in lens]
    vs = [rng.standard_normal((L, Hkv, D)) for L in lens]
    q = rng.standard_normal((3, 4, D))
    kc, vc, bt = _paged_from_dense(rng, ks, vs, B, NB)
    qsl = np.arange(4, dtype=np.int32)
    base = paged_attention_ref(q, kc, vc, bt, np.array(lens, np.int32), qsl, 0.3, B)
    relabel = rng.permutation(NB)
    kc2, vc2 = np.zeros_like(kc), np.zeros_like(vc)
    kc2[relabel], vc2[relabel] = kc, vc
    bt2 = relabel[bt].astype(np.int32)
    again = paged_attention_ref(q, kc2, vc2, bt2, np.array(lens, np.int32), qsl, 0.3, B)
    assert np.array_equal(base, again)


def test_single_key_returns_its_value():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 4, 16))
    k = rng.standard_normal((1, 2, 16))
    v = rng.standard_normal((1, 2, 16))
    out = dense_causal_ref(q, k, v, 0.7)
    assert np.array_equal(out[0], np.repeat(v[0], 2, axis=0))


def test_zero_query_averages_visible_values():
    rng = np.random.default_rng(2)
    L, n = 11, 3
    k = rng.standard_normal((L, 1, 8))
    v = rng.standard_normal((L, 1, 8))
    out = dense_causal_ref(np.zeros((n, 2, 8)), k, v, 0.5)
    for j in range(n):
        last = L - n + j
        assert np.allclose(out[j, 0], v[: last + 1, 0].mean(0), atol=1e-14)
        assert np.allclose(out[j, 1], v[: last + 1, 0].mean(0), atol=1e-14)


def test_sharp_softmax_selects_the_argmax_key():
    rng = np.random.default_rng(3)
    L, D = 9, 16
    k = rng.standard_normal((L, 1, D))
    v = rng.standard_normal((L, 1, D))
    q = rng.standard_normal((1, 1, D))
    out = dense_causal_ref(q, k, v, 1e4)
    assert np.allclose(out[0, 0], v[np.argmax(k[:, 0] @ q[0, 0]), 0], atol=1e-12)


def test_group_mapping_uses_consecutive_query_heads():
    # query heads 0,1 read KV head 0 and heads 2,3 read KV head 1 (not interleaved)
    rng = np.random.default_rng(4)
    k = rng.standard_normal((5, 2, 8))
    v = np.zeros((5, 2, 8))
    v[:, 1] = 1.0
    out = dense_causal_ref(rng.standard_normal((1, 4, 8)), k, v, 0.3)
    assert np.allclose(out[0, :2], 0.0) and np.allclose(out[0, 2:], 1.0)


def test_chunk_equals_sequence_of_single_queries():
    rng = np.random.default_rng(5)
    L, n = 23, 7
    k = rng.standard_normal((L, 2, 16))
    v = rng.standard_normal((L, 2, 16))
    q = rng.standard_normal((n, 4, 16))
    chunk = dense_causal_ref(q, k, v, 0.2)
    for j in range(n):
        upto = L - n + j + 1
        single = dense_causal_ref(q[j : j + 1], k[:upto], v[:upto], 0.2)
        assert np.array_equal(chunk[j], single[0])


def test_kv_write_closed_form_and_padding():
    rng = np.random.default_rng(6)
    NB, B, Hkv, D = 6, 4, 2, 8
    k = rng.integers(0, 2**16, (NB * B, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 2**16, (NB * B, Hkv, D), dtype=np.uint16)
    kc = np.zeros((NB, B, Hkv, D), np.uint16)
    vc = np.zeros_like(kc)
    slots = np.arange(NB * B)
    slots[5] = -1  # padding token: skipped
    kv_write_ref(kc, vc, k, v, slots, B)
    flat_k, flat_v = kc.reshape(-1, Hkv, D), vc.reshape(-1, Hkv, D)
    keep = slots >= 0
    assert np.array_equal(flat_k[keep], k[keep]) and np.array_equal(flat_v[keep], v[keep])
    assert not flat_k[5].any() and not flat_v[5].any()
    # reversed slots: token t lands in flat row N-1-t
    kc2 = np.zeros_like(kc)
    kv_write_ref(kc2, np.zeros_like(vc), k, v, np.arange(NB * B)[::-1], B)
    assert np.array_equal(kc2.reshape(-1, Hkv, D)[::-1], k)


def test_copy_blocks_closed_form():
    rng = np.random.default_rng(8)
    kc = rng.integers(0, 2**16, (8, 4, 2, 8), dtype=np.uint16)
    vc = rng.integers(0, 2**16, (8, 4, 2, 8), dtype=np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    copy_blocks_ref(kc, vc, [(1, 5), (5, 6), (2, 0)])  # applied in order: 6 gets 1's content
    want_k = k0.copy()
    want_k[5], want_k[6], want_k[0] = k0[1], k0[1], k0[2]
    want_v = v0.copy()
    want_v[5], want_v[6], want_v[0] = v0[1], v0[1], v0[2]
    assert np.array_equal(kc, want_k) and np.array_equal(vc, want_v)
    copy_blocks_ref(kc, vc, [])
    assert np.array_equal(kc, want_k)


def test_block_store_matches_dense_cache():
    rng = np.random.default_rng(9)
    B, Hkv, D = 4, 2, 8
    k = rng.standard_normal((10, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((10, Hkv, D)).astype(np.float32)
    slots = [9 * 4 + i for i in range(4)] + [2 * 4 + i for i in range(4)] + [7 * 4, 7 * 4 + 1]
    dense_k, dense_v = np.zeros((12, B, Hkv, D), np.float32), np.zeros((12, B, Hkv, D), np.float32)
    sk, sv = BlockStore(B, Hkv, D, np.float32), BlockStore(B, Hkv, D, np.float32)
    kv_write_ref(dense_k, dense_v, k, v, slots, B)
    kv_write_ref(sk, sv, k, v, slots, B)
    copy_blocks_ref(dense_k, dense_v, [(2, 4)])
    copy_blocks_ref(sk, sv, [(2, 4)])
    for b in sk:
        assert np.array_equal(sk[b], dense_k[b]) and np.array_equal(sv[b], dense_v[b])
    bt = np.array([[9, 4, 7]], np.int32)
    q = rng.standard_normal((1, 4, D)).astype(np.float32)
    qsl = np.array([0, 1], np.int32)
    a = paged_attention_ref(q, dense_k, dense_v, bt, np.array([10], np.int32), qsl, 0.3, B)
    b = paged_attention_ref(q, sk, sv, bt, np.array([10], np.int32), qsl, 0.3, B)
    assert np.array_equal(a, b)
