"""Swapping on the GPU: pa_swap_blocks between the GPU pool and a pinned CPU pool, and the
preemption workload (a group swapped out, its GPU blocks overwritten by other work, swapped
back in, then decoded) against the oracle.

Bars: block bytes bit-exact; attention |err| <= 1.5e-2 + 1e-2 * |ref| (bf16).
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import run_workload, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_161_gb300 as m

    m.read_device_errors(clear=True)
    return m


def _bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float8_e4m3fn])
def test_swap_blocks_both_directions_exact(pa, dtype):
    NB, NC, B, H, D = 24, 10, 16, 8, 128
    g = torch.Generator().manual_seed(3)
    if dtype == torch.float8_e4m3fn:
        gk = torch.randint(0, 126, (NB, B, H, D), generator=g, dtype=torch.uint8).view(dtype).cuda()
        gv = torch.randint(0, 126, (NB, B, H, D), generator=g, dtype=torch.uint8).view(dtype).cuda()
    else:
        gk = torch.randn((NB, B, H, D), generator=g).to(dtype).cuda()
        gv = torch.randn((NB, B, H, D), generator=g).to(dtype).cuda()
    ck = torch.zeros((NC, B, H, D), dtype=dtype).pin_memory()
    cv = torch.zeros((NC, B, H, D), dtype=dtype).pin_memory()
    out_pairs = torch.tensor([[5, 0], [17, 9], [2, 4], [23, 1]], dtype=torch.int64)
    pa.swap_blocks(gk, gv, ck, cv, out_pairs.cuda())
    torch.cuda.synchronize()
    gkb, gvb, ckb, cvb = _bytes(gk), _bytes(gv), _bytes(ck), _bytes(cv)
    for s, d in out_pairs.tolist():
        assert np.array_equal(ckb[d], gkb[s]) and np.array_equal(cvb[d], gvb[s])
    assert not ckb[[2, 3, 5, 6, 7, 8]].any()
    # back in, to other blocks; the mapping itself in pinned host memory this time
    in_pairs = torch.tensor([[0, 11], [9, 3], [4, 20], [1, 0]], dtype=torch.int64).pin_memory()
    before = _bytes(gk).copy()
    pa.swap_blocks(ck, cv, gk, gv, in_pairs)
    torch.cuda.synchronize()
    gk2, gv2 = _bytes(gk), _bytes(gv)
    for s, d in in_pairs.tolist():
        assert np.array_equal(gk2[d], ckb[s]) and np.array_equal(gv2[d], cvb[s])
    untouched = [b for b in range(NB) if b not in (11, 3, 20, 0)]
    assert np.array_equal(gk2[untouched], before[untouched])
    assert pa.read_device_errors(clear=True) == 0
    bad = torch.tensor([[0, NB], [1, 2]], dtype=torch.int64, device="cuda")
    pa.swap_blocks(ck, cv, gk, gv, bad)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == pa.PA_DEVERR["block_range"]
    assert np.array_equal(_bytes(gk)[2], ckb[1])  # the valid pair still ran


def _run(pa, wl):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    dw.run_step(st)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    return dw, st, torch_to_storage


def test_preemption_small_matches_oracle(pa):
    wl = workloads.preemption("small")
    dw, st, t2s = _run(pa, wl)
    assert sum(len(p) for ph in dw.phase_swaps for _, p in ph) > 0
    ref = run_workload(wl)
    for a, b in zip(dw.phase_slots, ref.phase_slots):
        assert np.array_equal(a, b)
    assert np.array_equal(t2s(dw.k_cache), ref.k_cache) and np.array_equal(t2s(dw.v_cache), ref.v_cache)
    err = np.abs(to_f64(t2s(st.out)) - ref.out)
    assert not (err > 1.5e-2 + 1e-2 * np.abs(ref.out)).any()


def test_preemption_full_swapped_group_sampled(pa):
    wl = workloads.preemption("full")
    dw, st, t2s = _run(pa, wl)
    pick = sorted(set(wl.meta["swapped_group"]) | {5, 30, 63})
    ref = run_workload(wl, eval_seqs=pick)
    out = to_f64(t2s(st.out))
    err = np.abs(out[pick] - ref.out[pick])
    assert not (err > 1.5e-2 + 1e-2 * np.abs(ref.out[pick])).any()
    kc = t2s(dw.k_cache)
    B = wl.spec.block_size
    for i in wl.meta["swapped_group"]:
        table = ref.block_table[i]
        for pos in range(0, int(ref.seq_lens[i]), 5):
            assert np.array_equal(kc[table[pos // B], pos % B], ref.k_cache[table[pos // B]][pos % B])


def test_swap_rejects_pageable_host_memory_before_launch(pa):
    """A pool in ordinary (pageable) host memory is refused by the library's pointer check,
    so no kernel ever dereferences it."""
    NB, B, H, D = 4, 16, 8, 128
    gk = torch.zeros((NB, B, H, D), dtype=torch.bfloat16, device="cuda")
    gv = torch.zeros_like(gk)
    host = np.zeros((NB, B, H, D), np.uint16)  # pageable
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device="cuda")
    st = pa.lib.pa_swap_blocks(gk.data_ptr(), gv.data_ptr(), host.ctypes.data, host.ctypes.data,
                               pairs.data_ptr(), 1, NB, NB, B, H, D, pa.PA_BF16, None)
    assert st == 1
    with pytest.raises(ValueError):
        pa.swap_blocks(gk, gv, torch.zeros((NB, B, H, D), dtype=torch.bfloat16),
                       torch.zeros((NB, B, H, D), dtype=torch.bfloat16), pairs)
