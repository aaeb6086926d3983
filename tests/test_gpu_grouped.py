"""pa_attention_grouped (a shared prefix read once per group) against the oracle and
against pa_attention on the same batch.

Bars: attention |err| <= 1.5e-2 + 1e-2 * |ref| (bf16) and the diagnostic bound of
tests/errmodel.py against the float64 oracle; against pa_attention within twice the pass
bar (both round P to bf16, in different orders).
"""
import numpy as np
import pytest
import torch

import workloads
from errmodel import assert_close_bf16, batch_sigma
from oracle import run_workload, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_161_gb300 as m

    m.read_device_errors(clear=True)
    return m


def _close(got, ref, what, k=1.0):
    err = np.abs(to_f64(got) - ref)
    bad = err > k * (1.5e-2 + 1e-2 * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, max err {err.max()}"


def _step(pa, wl):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    plain = dw.run_step(st).clone()  # copies, writes, pa_attention
    torch.cuda.synchronize()
    return dw, st, plain, torch_to_storage


def _grouped(pa, dw, st, wl, seq_group, group_range, shared_len):
    out = torch.empty_like(st.q)
    dev = st.q.device
    pa.attention_grouped(out, st.q, dw.k_cache, dw.v_cache, st.block_table, st.seq_lens, st.query_start_loc,
                         torch.from_numpy(seq_group).to(dev), torch.from_numpy(group_range).to(dev),
                         torch.from_numpy(shared_len).to(dev), max_seq_len=st.max_seq_len, scale=wl.spec.scale)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    return out


@pytest.mark.parametrize("max_members", [4, 3, 2])
def test_grouped_shared_prefix_small(pa, max_members):
    wl = workloads.build(4, "small")
    dw, st, plain, t2s = _step(pa, wl)
    seqs = [s for s, _ in wl.step.batch]
    sg, gr, sl = dw.bm.batch_groups(seqs, max_members)
    assert len(gr) > 0 and (sl >= 16).any()
    out = _grouped(pa, dw, st, wl, sg, gr, sl)
    ref = run_workload(wl)
    _close(t2s(out), ref.out, "grouped vs oracle")
    sig = batch_sigma(ref, range(len(ref.seq_lens)), wl.spec.scale, wl.spec.block_size)
    assert_close_bf16(to_f64(t2s(out)), ref.out, sig, "grouped vs oracle")
    _close(t2s(out), to_f64(t2s(plain)), "grouped vs pa_attention", k=2.0)


def test_grouped_full_size_all_requests(pa):
    wl = workloads.build(4)
    dw, st, plain, t2s = _step(pa, wl)
    seqs = [s for s, _ in wl.step.batch]
    sg, gr, sl = dw.bm.batch_groups(seqs, 4)
    assert len(gr) == wl.meta["prompts"]
    out = t2s(_grouped(pa, dw, st, wl, sg, gr, sl))
    ref = run_workload(wl)
    sig = batch_sigma(ref, range(len(ref.seq_lens)), wl.spec.scale, wl.spec.block_size)
    assert_close_bf16(to_f64(out), ref.out, sig, "grouped vs oracle")
    _close(out, to_f64(t2s(plain)), "grouped vs pa_attention", k=2.0)


@pytest.mark.parametrize("P,prompt_len,tail_hi,seed", [(2, 200, 300, 161041), (5, 33, 70, 161042)])
def test_grouped_long_member_tails(pa, P, prompt_len, tail_hi, seed):
    """Members whose own chunks outnumber the shared ones, in a batch smaller than the
    grid: a group's segment (its shared chunks, then each member's own) spreads over many
    CTAs, some of them with empty ranges, and a member's result merges dozens of pieces."""
    wl = workloads.shared_prefix(P, prompt_len, 4, tail_hi, seed)
    dw, st, plain, t2s = _step(pa, wl)
    seqs = [s for s, _ in wl.step.batch]
    sg, gr, sl = dw.bm.batch_groups(seqs, 4)
    assert len(gr) == P
    out = t2s(_grouped(pa, dw, st, wl, sg, gr, sl))
    ref = run_workload(wl)
    sig = batch_sigma(ref, range(len(ref.seq_lens)), wl.spec.scale, wl.spec.block_size)
    assert_close_bf16(to_f64(out), ref.out, sig, "grouped vs oracle")
    _close(out, to_f64(t2s(plain)), "grouped vs pa_attention", k=2.0)


def test_grouped_degenerate_groups_match_plain(pa):
    """No groups; a member whose seq_group disagrees with its range (it runs on its own);
    groups too wide for 16 matrix rows (G = 8 x 4 members: they run ungrouped)."""
    wl = workloads.build(4, "small")
    dw, st, plain, t2s = _step(pa, wl)
    seqs = [s for s, _ in wl.step.batch]
    z = np.zeros(0, np.int32)
    out = _grouped(pa, dw, st, wl, np.full(len(seqs), -1, np.int32), z.reshape(0, 2), z)
    _close(t2s(out), to_f64(t2s(plain)), "no groups", k=2.0)
    sg, gr, sl = dw.bm.batch_groups(seqs, 4)
    sg = sg.copy()
    sg[1] = -1
    out = _grouped(pa, dw, st, wl, sg, gr, sl)
    _close(t2s(out), to_f64(t2s(plain)), "inconsistent member", k=2.0)
    spec = workloads.Spec("bf16", 32, 4, 128, 16, 0.088)  # G = 8
    wl8 = workloads.custom(spec, [40, 40, 40, 40], [1, 1, 1, 1], name="g8")
    dw8, st8, plain8, _ = _step(pa, wl8)
    sg8 = np.zeros(4, np.int32)
    out8 = _grouped(pa, dw8, st8, wl8, sg8, np.array([[0, 4]], np.int32), np.array([32], np.int32))
    _close(t2s(out8), to_f64(t2s(plain8)), "16-row cap", k=2.0)
