"""pa_attention_fixed_scratch, the attention entry point for callers that cannot allocate
device memory (a serving loop whose KV pool already owns the GPU's memory, a plugin without
access to its host's allocator, a binding with no device allocator): instead of a caller
workspace it uses a fixed scratch array inside the library.

Checked through the C ABI against pa_attention (caller workspace) on the same inputs, on
two calls in a row: the second call starts from whatever the first left in the shared
scratch. This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from oracle import to_f64

pytestmark = pytest.mark.gpu

FIXED_SCRATCH_BYTES = 16 << 20


def _entry(pa):
    f = pa.lib.pa_attention_fixed_scratch
    p, i, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.restype = i
    f.argtypes = [p, p, p, p, p, i, p, p, i, i, i, i, i, i, i, i, i64, ctypes.c_float, i, p]
    return f


def _call(f, out, q, kc, vc, bt, lens, qsl, max_q, max_s, scale):
    NB, B, Hkv, D = kc.shape
    dt = 0 if q.dtype == torch.float32 else 1
    return f(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), int(bt.shape[1]),
             lens.data_ptr(), qsl.data_ptr(), int(lens.shape[0]), int(q.shape[0]), int(max_q), int(max_s),
             int(q.shape[1]), Hkv, D, B, NB, float(scale), dt, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("cfg,size", [(3, "small"), (3, "full"), (5, "small"), (5, "full"), (1, "full"), (2, "small")])
def test_matches_workspace_entry_point_on_two_calls(cfg, size):
    import paged_kv_cache_161_gb300 as pa
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    wl = workloads.build(cfg, size)
    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    dw.run_step(st)  # pa_kv_write + pa_attention with a caller workspace
    torch.cuda.synchronize()
    ref = to_f64(torch_to_storage(st.out))
    f = _entry(pa)
    for _ in range(2):
        out = torch.full_like(st.q, float("nan"))
        status = _call(f, out, st.q, dw.k_cache, dw.v_cache, st.block_table, st.seq_lens, st.query_start_loc,
                       st.max_query_len, st.max_seq_len, wl.spec.scale)
        assert status == 0, pa.lib.pa_status_string(status)
        torch.cuda.synchronize()
        got = to_f64(torch_to_storage(out))
        err = np.abs(got - ref)
        if wl.spec.dtype == "f32":
            assert err.max() <= 2e-5
        else:
            assert (err <= 1.5e-2 + 1e-2 * np.abs(ref)).all()
    assert pa.read_device_errors(clear=True) == 0


def test_rejects_batch_needing_more_than_the_fixed_scratch():
    import paged_kv_cache_161_gb300 as pa

    S, Hq, Hkv, D, B = 4096, 32, 8, 128, 16
    assert pa.attention_workspace_size(S, Hq, Hkv, D) > FIXED_SCRATCH_BYTES
    dev = "cuda"
    kc = torch.zeros((8, B, Hkv, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    q = torch.zeros((S, Hq, D), dtype=torch.bfloat16, device=dev)
    out = torch.zeros_like(q)
    bt = torch.zeros((S, 1), dtype=torch.int32, device=dev)
    lens = torch.ones(S, dtype=torch.int32, device=dev)
    qsl = torch.arange(S + 1, dtype=torch.int32, device=dev)
    f = _entry(pa)
    status = _call(f, out, q, kc, vc, bt, lens, qsl, 1, 1, 0.088)
    assert status == 3  # PA_ERR_WORKSPACE: nothing was enqueued
    torch.cuda.synchronize()
    assert not out.any()
