"""pa_attention_fixed_scratch, the attention entry point for callers that cannot allocate
device memory (a serving loop whose KV pool already owns the GPU's memory, a plugin without
access to its host's allocator, a binding with no device allocator): instead of a caller
workspace it uses a fixed scratch array inside the library.

Checked through the C ABI against pa_attention (caller workspace) on the same inputs, on
two calls in a row: the second call starts from whatever the first left in the shared
scratch. Each call's output is also checked directly against the float64 oracle (the pass
bar, and for bf16 the diagnostic bound of tests/errmodel.py): every request of the reduced
workloads, and for the full-size GQA and mixed batches the longest request, every
chunked-prefill request and a seeded sample of the rest. This file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from errmodel import assert_close_bf16, batch_sigma
from oracle import run_workload, to_f64

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
    n = len(wl.step.batch)
    if size == "full":
        lens = wl.meta["final_lens"]
        pick = {int(np.argmax(lens))} | {i for i, (_, q) in enumerate(wl.step.batch) if q != 1}
        pick |= set(int(i) for i in np.random.default_rng(cfg).choice(n, min(12, n), replace=False))
        pick = sorted(pick)
    else:
        pick = list(range(n))
    oref = run_workload(wl, eval_seqs=None if size != "full" else pick)
    qsl = oref.query_start_loc
    rows = np.concatenate([np.arange(qsl[i], qsl[i + 1]) for i in pick])
    sig = batch_sigma(oref, pick, wl.spec.scale, wl.spec.block_size)[rows] if wl.spec.dtype == "bf16" else None
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
            assert np.abs(got[rows] - oref.out[rows]).max() <= 2e-5
        else:
            assert (err <= 1.5e-2 + 1e-2 * np.abs(ref)).all()
            assert_close_bf16(got[rows], oref.out[rows], sig, f"fixed scratch vs oracle, {wl.name}")
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
