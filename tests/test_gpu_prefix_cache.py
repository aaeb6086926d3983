"""Prefix caching on the GPU: requests that reuse a cached system prompt run chunked
prefill over the reused blocks; cache bytes and outputs must match the oracle.

Bars: cache contents bit-exact; attention |err| <= 1.5e-2 + 1e-2 * |ref| (bf16).
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


def _close(got, ref, what):
    err = np.abs(to_f64(got) - ref)
    bad = err > 1.5e-2 + 1e-2 * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance"


def _device_step(pa, wl):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    dw.run_step(st, fused=True)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    return dw, st, torch_to_storage


@pytest.mark.parametrize("caching", [True, False])
def test_system_prompt_small_matches_oracle(pa, caching):
    wl = workloads.system_prompt("small", caching=caching)
    dw, st, t2s = _device_step(pa, wl)
    ref = run_workload(wl)
    assert np.array_equal(t2s(dw.k_cache), ref.k_cache) and np.array_equal(t2s(dw.v_cache), ref.v_cache)
    assert np.array_equal(st.query_start_loc.cpu().numpy(), ref.query_start_loc)
    _close(t2s(st.out), ref.out, wl.name)


def test_system_prompt_full_cached_sampled(pa):
    """64 requests reusing a 2032-token cached prefix; sampled requests vs the oracle, and
    every request's reused prefix reads back the warm request's K/V."""
    wl = workloads.system_prompt("full", caching=True)
    dw, st, t2s = _device_step(pa, wl)
    pick = [0, 17, 40, 63]
    ref = run_workload(wl, eval_seqs=pick)
    assert np.array_equal(st.query_start_loc.cpu().numpy(), ref.query_start_loc)
    qsl = ref.query_start_loc
    rows = np.concatenate([np.arange(qsl[i], qsl[i + 1]) for i in pick])
    out = t2s(st.out)
    _close(out[rows], ref.out[rows], wl.name)
    kc = t2s(dw.k_cache)
    B, P = wl.spec.block_size, wl.meta["system_len"]
    k_sys, _ = wl.kv(wl.meta["requests"], 0, P)
    table = st.block_table.cpu().numpy()
    for i in range(wl.meta["requests"]):
        for p in range(0, (P // B) * B, 97):
            assert np.array_equal(kc[table[i, p // B], p % B], k_sys[p])


def test_cached_rows_agree_with_uncached_rows(pa):
    """The rows a cached request computes equal (within the bf16 bar of each other) the
    same positions' rows of the uncached run."""
    outs = {}
    for caching in (True, False):
        wl = workloads.system_prompt("small", caching=caching)
        dw, st, t2s = _device_step(pa, wl)
        outs[caching] = (to_f64(t2s(st.out)), st.query_start_loc.cpu().numpy(), st.seq_lens.cpu().numpy())
    (oc, qc, lc), (ou, qu, lu) = outs[True], outs[False]
    assert np.array_equal(lc, lu)
    for i in range(len(lc)):
        n = qc[i + 1] - qc[i]
        a, b = oc[qc[i]:qc[i + 1]], ou[qu[i + 1] - n:qu[i + 1]]
        assert np.all(np.abs(a - b) <= 2 * (1.5e-2 + 1e-2 * np.abs(b)))
