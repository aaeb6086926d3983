"""CUDA path vs the float64 oracle, element by element, through the C ABI.

Bars: cache writes, block copies, slot mappings and copy pairs bit-exact; attention
max|err| <= 2e-5 for fp32 inputs; for bf16 inputs the pass bar |err| <= 1.5e-2 + 1e-2 |ref|
and, beside it, the diagnostic bound of tests/errmodel.py (the kernels' own rounding:
|err| <= 2^-8 (1 + 2^-7) |ref| + 4 u sigma + 1e-5), which a dropped block or stage fails
even at 8192 keys. At full size every request of the batch is evaluated, so a request cut
between CTAs anywhere, the longest one and every chunked prefill are all covered.
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


def _close(got, ref, dtype, what, sigma=None):
    got = to_f64(got)
    err = np.abs(got - ref)
    if dtype == "f32":
        assert np.max(err) <= 2e-5, f"{what}: max err {np.max(err)}"
    elif sigma is not None:
        assert_close_bf16(got, ref, sigma, what)
    else:
        bound = 1.5e-2 + 1e-2 * np.abs(ref)
        bad = err > bound
        assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, worst {np.max(err - bound)}"


def _sigma(wl, ref, seqs=None):
    """Error scale of the diagnostic bound for the evaluated rows (bf16 workloads)."""
    if wl.spec.dtype != "bf16":
        return None
    seqs = range(len(ref.seq_lens)) if seqs is None else seqs
    return batch_sigma(ref, seqs, wl.spec.scale, wl.spec.block_size)


def _run(pa, wl, eval_seqs=None):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    dw.run_step(st)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    ref = run_workload(wl, eval_seqs=eval_seqs)
    out = torch_to_storage(st.out)
    return dw, st, out, ref, torch_to_storage


def _check_accounting(dw, ref):
    assert len(dw.phase_slots) == len(ref.phase_slots)
    for a, b in zip(dw.phase_slots, ref.phase_slots):
        assert np.array_equal(a, b)
    for a, b in zip(dw.phase_copies, ref.phase_copies):
        assert a.tolist() == [list(p) for p in b]


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_small_workload_matches_oracle(pa, cfg):
    wl = workloads.build(cfg, "small")
    dw, st, out, ref, t2s = _run(pa, wl)
    _check_accounting(dw, ref)
    assert np.array_equal(t2s(dw.k_cache), ref.k_cache)
    assert np.array_equal(t2s(dw.v_cache), ref.v_cache)
    _close(out, ref.out, wl.spec.dtype, wl.name, _sigma(wl, ref))


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_full_size_all_requests(pa, cfg):
    """The workloads at full size (the bench's launch configuration for the GQA batch):
    the whole caches bit-exact and every request's rows against the oracle."""
    wl = workloads.build(cfg)
    dw, st, out, ref, t2s = _run(pa, wl)
    _check_accounting(dw, ref)
    kc, vc = t2s(dw.k_cache), t2s(dw.v_cache)
    assert np.array_equal(kc, ref.k_cache)
    assert np.array_equal(vc, ref.v_cache)
    _close(out, ref.out, wl.spec.dtype, wl.name, _sigma(wl, ref))


def test_output_bits_independent_of_physical_placement(pa):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    outs = []
    for perm_seed in (None, 1, 2):
        wl = workloads.build(3, "small")
        if perm_seed is not None:
            wl.free_order = np.random.default_rng(perm_seed).permutation(wl.num_blocks).astype(np.int32)
        dw = DeviceWorkload(wl)
        dw.run_setup()
        st = dw.prepare_step()
        dw.run_step(st)
        torch.cuda.synchronize()
        outs.append(torch_to_storage(st.out))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


EDGE = [
    # (name, spec, ctx, q_lens)
    ("single_token", workloads.Spec("bf16", 32, 8, 128, 16, 0.088), [0, 0, 5], [1, 1, 1]),
    ("block_multiples", workloads.Spec("bf16", 32, 8, 128, 16, 0.088), [15, 31, 47, 16, 32], [1, 1, 1, 1, 1]),
    ("one_long_sequence", workloads.Spec("bf16", 32, 8, 128, 16, 0.088), [20000], [1]),
    ("empty_query_rows", workloads.Spec("bf16", 32, 8, 128, 16, 0.088), [10, 40, 3], [1, 0, 2]),
    ("fp32_d128_g2", workloads.Spec("f32", 8, 4, 128, 16, 0.1), [33, 70, 1], [1, 1, 3]),
    ("bf16_d64_g8_b32", workloads.Spec("bf16", 16, 2, 64, 32, 0.125), [100, 5, 64], [1, 1, 4]),
    ("fp32_b1_g1", workloads.Spec("f32", 2, 2, 64, 1, 0.125), [9, 17], [1, 2]),
    ("bf16_b8_mqa", workloads.Spec("bf16", 4, 1, 128, 8, 0.088), [23, 8, 70], [1, 1, 1]),
    ("many_short", workloads.Spec("bf16", 32, 8, 128, 16, 0.088), list(range(1, 300)), [1] * 299),
    # chunked prefill on the tensor cores (bf16): group sizes, head dims, block sizes
    ("prefill_g4_b16", workloads.Spec("bf16", 32, 8, 128, 16, 0.088), [0, 100, 300, 7], [200, 77, 5, 1]),
    ("prefill_g1_b64", workloads.Spec("bf16", 8, 8, 128, 64, 0.088), [50, 0], [130, 300]),
    ("prefill_g2_d64_b128", workloads.Spec("bf16", 8, 4, 64, 128, 0.125), [129, 0], [40, 256]),
    ("prefill_g8_b8", workloads.Spec("bf16", 32, 4, 128, 8, 0.088), [17, 0], [60, 2]),
    ("prefill_long_prior", workloads.Spec("bf16", 32, 8, 128, 16, 0.088), [3000], [300]),
    # softmax scale 1 (logits with a standard deviation of ~11): the running max keeps
    # jumping by more than 2^8 deep into a sequence, so the decode and prefill kernels move
    # their reference max and rescale O mid-sequence, not only at the first keys
    ("sharp_softmax_mixed", workloads.Spec("bf16", 32, 8, 128, 16, 1.0), [700, 2500, 0, 90], [1, 1, 260, 1]),
]


@pytest.mark.parametrize("name,spec,ctx,q_lens", EDGE, ids=[e[0] for e in EDGE])
def test_edge_cases(pa, name, spec, ctx, q_lens):
    wl = workloads.custom(spec, ctx, q_lens, name=name)
    dw, st, out, ref, t2s = _run(pa, wl)
    _check_accounting(dw, ref)
    assert np.array_equal(t2s(dw.k_cache), ref.k_cache)
    qsl = ref.query_start_loc
    rows = np.concatenate([np.arange(qsl[i], qsl[i + 1]) for i in range(len(q_lens))])
    if len(rows):
        sig = _sigma(wl, ref)
        _close(out[rows], ref.out[rows], spec.dtype, name, None if sig is None else sig[rows])


def test_prefill_output_only_16_byte_aligned(pa):
    """An output buffer that is 16- but not 32-byte aligned (the ABI's minimum) takes the
    prefill epilogue's 16-byte stores; the bits equal those written to an aligned buffer."""
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    wl = workloads.custom(workloads.Spec("bf16", 32, 8, 128, 16, 0.088), [0, 300, 40], [200, 70, 1], name="a16")
    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    dw.run_step(st)
    torch.cuda.synchronize()
    T, H, D = st.q.shape
    flat = torch.full((T * H * D + 8,), float("nan"), dtype=torch.bfloat16, device=st.q.device)
    out16 = flat[8:].view(T, H, D)  # 16 bytes past a 256-byte aligned allocation
    assert out16.data_ptr() % 32 == 16
    pa.attention(out16, st.q, dw.k_cache, dw.v_cache, st.block_table, st.seq_lens, st.query_start_loc,
                 max_query_len=st.max_query_len, max_seq_len=st.max_seq_len, scale=wl.spec.scale,
                 workspace=st.workspace)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    assert torch.equal(out16, st.out)


def test_kv_write_padding_and_bad_slots(pa):
    dev = "cuda"
    NB, B, H, D = 8, 16, 8, 128
    kc = torch.zeros((NB, B, H, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    k = torch.randn((4, H, D), device=dev).to(torch.bfloat16)
    v = torch.randn((4, H, D), device=dev).to(torch.bfloat16)
    slots = torch.tensor([3, -1, 17, NB * B + 5], dtype=torch.int64, device=dev)
    pa.kv_write(k, v, kc, vc, slots)
    torch.cuda.synchronize()
    flags = pa.read_device_errors(clear=True)
    assert flags == pa.PA_DEVERR["slot_range"]
    flat_k, flat_v = kc.view(-1, H, D), vc.view(-1, H, D)
    assert torch.equal(flat_k[3], k[0]) and torch.equal(flat_k[17], k[2])
    assert torch.equal(flat_v[3], v[0]) and torch.equal(flat_v[17], v[2])
    others = [i for i in range(NB * B) if i not in (3, 17)]
    assert not flat_k[others].any() and not flat_v[others].any()


def test_copy_blocks_exact_and_empty(pa):
    dev = "cuda"
    NB, B, H, D = 16, 16, 8, 128
    kc = torch.randn((NB, B, H, D), device=dev).to(torch.bfloat16)
    vc = torch.randn((NB, B, H, D), device=dev).to(torch.bfloat16)
    k0, v0 = kc.clone(), vc.clone()
    pa.copy_blocks(kc, vc, torch.zeros((0, 2), dtype=torch.int64, device=dev))
    torch.cuda.synchronize()
    assert torch.equal(kc, k0)
    pairs = torch.tensor([[1, 9], [4, 2], [7, 15]], dtype=torch.int64, device=dev)
    pa.copy_blocks(kc, vc, pairs)
    torch.cuda.synchronize()
    want_k, want_v = k0.clone(), v0.clone()
    for s, d in pairs.tolist():
        want_k[d], want_v[d] = k0[s], v0[s]
    assert torch.equal(kc, want_k) and torch.equal(vc, want_v)
    bad = torch.tensor([[1, NB], [2, 3]], dtype=torch.int64, device=dev)
    pa.copy_blocks(kc, vc, bad)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == pa.PA_DEVERR["block_range"]
    assert torch.equal(kc[3], want_k[2]) and torch.equal(vc[3], want_v[2])  # the valid pair still ran
    assert torch.equal(kc[1], want_k[1])


def test_repeated_steps_are_deterministic(pa):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    wl = workloads.build(3, "small")
    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    a = dw.run_step(st).clone()
    b = dw.run_step(st).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
