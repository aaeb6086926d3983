"""Requests cut between CTAs of the split-K decode kernel, merged by their log-sum-exps.

- Outputs against the oracle for batches whose cuts fall everywhere: one short request
  (a few units spread over CTAs far apart, empty CTAs in between), one long request (tens
  of pieces), a mix of lengths; GQA, MHA, head_dim 64, 8 query heads per KV head and
  block size 8, bf16, through pa_write_attention (the KV write fused in); and an E4M3 cache.
- One workspace reused across batches of different shapes (never cleared, holding the
  previous call's pieces) gives the same bits as a fresh workspace per call.

Bars against the float64 oracle (bf16 outputs): |err| <= 1.5e-2 + 1e-2 * |ref|, and for
bf16 caches also the diagnostic bound of tests/errmodel.py, which a piece lost or merged
twice fails even for the 20000-key request.
"""
import numpy as np
import pytest
import torch

import workloads
from errmodel import assert_close_bf16, batch_sigma
from oracle import run_workload, to_f64

pytestmark = pytest.mark.gpu

GQA = workloads.Spec("bf16", 32, 8, 128, 16, 128 ** -0.5)
MHA = workloads.Spec("bf16", 32, 32, 128, 16, 128 ** -0.5)
D64 = workloads.Spec("bf16", 16, 4, 64, 16, 64 ** -0.5)
G8 = workloads.Spec("bf16", 32, 4, 128, 16, 128 ** -0.5)   # query rows too large for shared-memory slots
B8 = workloads.Spec("bf16", 32, 8, 128, 8, 128 ** -0.5)    # two 8-token boxes per stage
CASES = {
    "one_short": [39],
    "one_long": [20000],
    "mixed": [8191, 5, 3000, 17, 16, 1, 250, 4097],
}


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_161_gb300 as m

    m.read_device_errors(clear=True)
    return m


def _close(got, ref, what):
    err = np.abs(to_f64(got) - ref)
    bad = err > 1.5e-2 + 1e-2 * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, max err {err.max()}"


def _run(pa, wl, ws=None, fused=False):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    if ws is not None:
        st.workspace = ws
    out = dw.run_step(st, fused=fused and not dw.fp8).clone()
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    return torch_to_storage(out), st.workspace


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("spec_name", ["gqa", "mha", "d64", "g8", "b8"])
def test_cut_requests_match_oracle(pa, case, spec_name):
    spec = {"gqa": GQA, "mha": MHA, "d64": D64, "g8": G8, "b8": B8}[spec_name]
    ctx = CASES[case]
    wl = workloads.custom(spec, ctx, [1] * len(ctx), name=f"{case}_{spec_name}")
    out, _ = _run(pa, wl, fused=True)
    ref = run_workload(wl)
    sig = batch_sigma(ref, range(len(ctx)), spec.scale, spec.block_size)
    assert_close_bf16(to_f64(out), ref.out, sig, wl.name)


@pytest.mark.parametrize("case", ["one_short", "mixed"])
def test_cut_requests_fp8_cache(pa, case):
    ctx = CASES[case]
    wl = workloads.with_fp8_cache(workloads.custom(GQA, ctx, [1] * len(ctx), name=case), k_scale=2.0 ** -6,
                                  v_scale=0.0123)
    out, _ = _run(pa, wl)
    _close(out, run_workload(wl).out, wl.name)


def test_one_workspace_reused_across_shapes(pa):
    """One workspace of arbitrary contents serves decode batches and a prefill batch whose
    ~580 tensor-core pairs outnumber the CTAs (the prefill's pair counter lives in it)."""
    wls = [workloads.custom(GQA, CASES["mixed"], [1] * 8, name="a"),
           workloads.custom(MHA, [5000, 39, 1200], [1, 1, 1], name="b"),
           workloads.custom(D64, CASES["one_long"], [1], name="c"),
           workloads.build(3, "small"),
           workloads.custom(GQA, [0, 2000, 700, 0, 3000, 100], [1500, 600, 900, 1200, 300, 1], name="p")]
    need = max(pa.attention_workspace_size(len(wl.step.batch), wl.spec.num_heads, wl.spec.num_kv_heads,
                                           wl.spec.head_dim) for wl in wls)
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda")  # arbitrary contents
    for rep in range(2):
        for wl in wls:
            fresh, _ = _run(pa, wl)
            shared, _ = _run(pa, wl, ws=ws, fused=rep == 1)
            assert np.array_equal(fresh, shared), wl.name
