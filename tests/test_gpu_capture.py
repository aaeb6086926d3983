"""Mixed batches (decode and chunked-prefill rows in one call) captured into a CUDA graph.

While the caller's stream is being captured, pa_attention keeps every kernel on that stream
(the internal side stream is shared by all callers of a device and must not join a
capture). Checked here: the capture succeeds, a replay gives the oracle's result within the
pass bar and the diagnostic bound, two replays give identical bits, and an eager mixed call
made after the capture still takes the side-by-side path and agrees with the oracle.
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


@pytest.mark.parametrize("fused", [False, True])
def test_captured_mixed_call_matches_oracle(pa, fused):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    wl = workloads.build(5, "small")
    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    assert st.max_query_len >= 2 and (st.query_start_loc.diff() == 1).any()  # both kinds of rows
    sp = wl.spec
    if not fused:
        pa.kv_write(st.k_new, st.v_new, dw.k_cache, dw.v_cache, st.slot_mapping)
    torch.cuda.synchronize()

    def call():
        if fused:  # the write of the chunk's tokens is part of the captured call
            pa.write_attention(st.out, st.q, st.k_new, st.v_new, st.slot_mapping, dw.k_cache, dw.v_cache,
                               st.block_table, st.seq_lens, st.query_start_loc, max_query_len=st.max_query_len,
                               max_seq_len=st.max_seq_len, scale=sp.scale, workspace=st.workspace)
        else:
            pa.attention(st.out, st.q, dw.k_cache, dw.v_cache, st.block_table, st.seq_lens, st.query_start_loc,
                         max_query_len=st.max_query_len, max_seq_len=st.max_seq_len, scale=sp.scale,
                         workspace=st.workspace)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    outs = []
    for _ in range(2):
        st.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        outs.append(torch_to_storage(st.out))
    assert pa.read_device_errors(clear=True) == 0
    assert np.array_equal(outs[0], outs[1])
    ref = run_workload(wl)
    sig = batch_sigma(ref, range(len(ref.seq_lens)), sp.scale, sp.block_size)
    assert_close_bf16(to_f64(outs[0]), ref.out, sig, "captured mixed call")

    st.out.fill_(float("nan"))  # an eager call after the capture (side by side again)
    call()
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    assert_close_bf16(to_f64(torch_to_storage(st.out)), ref.out, sig, "eager mixed call after a capture")
