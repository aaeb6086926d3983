"""FP8 (E4M3) KV cache on the GPU against the oracle.

Bars: the quantised cache bytes bit-exact (E4M3(x / scale), binary32 division, round to
nearest even, saturation); attention over the cache |err| <= 1.5e-2 + 1e-2 * |ref|
against the oracle's float64 attention over the dequantised values. Chunked-prefill rows
over an E4M3 cache run on the tensor cores (codes converted to f16 tiles in shared
memory): the mixed batch at full size (every request), the system-prompt batches with and
without prefix caching, and edge cases of group size, block size and context.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import quantize, run_workload, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_161_gb300 as m

    m.read_device_errors(clear=True)
    return m


def _close(got, ref, what):
    err = np.abs(to_f64(got) - ref)
    bad = err > 1.5e-2 + 1e-2 * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, max err {err.max()}"


def _codes(t):
    return t.detach().cpu().view(torch.uint8).numpy()


@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("scale", [2.0 ** -6, 0.0123])
def test_kv_write_fp8_bit_exact(pa, in_dtype, scale):
    """Values across E4M3's whole range (subnormal codes, ties, saturation, signed zeros),
    a padding slot and an out-of-range slot."""
    NB, B, H, D = 8, 16, 8, 128
    g = torch.Generator().manual_seed(5)
    T = 6
    x = torch.randn((2, T, H, D), generator=g) * torch.tensor([1e-4, 1e-2, 1.0, 3.0, 30.0, 1e3]).view(1, T, 1, 1)
    x[0, 0, 0, :4] = torch.tensor([0.0, -0.0, 448.0 * scale, -1e9])
    k, v = x[0].to(in_dtype).cuda(), x[1].to(in_dtype).cuda()
    kc = torch.zeros((NB, B, H, D), dtype=torch.float8_e4m3fn, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.tensor([0, 17, -1, 40, 127, NB * B + 3], dtype=torch.int64, device="cuda")
    pa.kv_write_fp8(k, v, kc, vc, slots, scale, scale)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == pa.PA_DEVERR["slot_range"]
    kf, vf = _codes(kc).reshape(NB * B, H, D), _codes(vc).reshape(NB * B, H, D)
    k32, v32 = k.float().cpu().numpy(), v.float().cpu().numpy()
    for t, s in enumerate(slots.tolist()):
        if 0 <= s < NB * B:
            assert np.array_equal(kf[s], quantize(k32[t], scale)), t
            assert np.array_equal(vf[s], quantize(v32[t], scale)), t
    written = {0, 17, 40, 127}
    others = [i for i in range(NB * B) if i not in written]
    assert not kf[others].any() and not vf[others].any()


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_fp8_small_workloads_match_oracle(pa, cfg):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    base = workloads.build(cfg, "small")
    if base.spec.dtype != "bf16":
        pytest.skip("E4M3 caches take bf16 queries")
    wl = workloads.with_fp8_cache(base, k_scale=2.0 ** -6, v_scale=0.0123)
    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    dw.run_step(st)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    ref = run_workload(wl)
    assert np.array_equal(torch_to_storage(dw.k_cache), ref.k_cache)
    assert np.array_equal(torch_to_storage(dw.v_cache), ref.v_cache)
    _close(torch_to_storage(st.out), ref.out, wl.name)


def test_fp8_full_size_gqa_decode_sampled(pa):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    wl = workloads.with_fp8_cache(workloads.build(3))
    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    dw.run_step(st)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    lens = np.array(wl.meta["final_lens"])
    pick = sorted({0, len(lens) - 1, int(np.argmax(lens)), int(np.argmin(lens)), 37, 101, 200})
    ref = run_workload(wl, eval_seqs=pick)
    out = torch_to_storage(st.out)
    _close(out[pick], ref.out[pick], wl.name)
    kc = torch_to_storage(dw.k_cache)
    B = wl.spec.block_size
    for i in pick:
        table = ref.block_table[i]
        for pos in range(0, int(ref.seq_lens[i]), 7):
            assert np.array_equal(kc[table[pos // B], pos % B], ref.k_cache[table[pos // B]][pos % B])


def test_fp8_decode_close_to_bf16_decode(pa):
    """The quantisation error itself: E4M3 keeps 3 mantissa bits, so outputs over the FP8
    cache stay within a few per cent of the bf16 cache's (a sanity bound, not parity)."""
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    outs = []
    for wl in (workloads.build(3, "small"), workloads.with_fp8_cache(workloads.build(3, "small"))):
        dw = DeviceWorkload(wl)
        dw.run_setup()
        st = dw.prepare_step()
        outs.append(to_f64(torch_to_storage(dw.run_step(st))))
    torch.cuda.synchronize()
    a, b = outs
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert rel < 0.05, rel


def test_fp8_copy_blocks_and_argument_checks(pa):
    NB, B, H, D = 8, 16, 8, 128
    kc = torch.randint(0, 126, (NB, B, H, D), dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    vc = torch.randint(0, 126, (NB, B, H, D), dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    k0, v0 = _codes(kc).copy(), _codes(vc).copy()
    pa.copy_blocks(kc, vc, torch.tensor([[1, 6], [3, 0]], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    k1, v1 = _codes(kc), _codes(vc)
    assert np.array_equal(k1[6], k0[1]) and np.array_equal(v1[0], v0[3]) and np.array_equal(k1[2], k0[2])
    q = torch.zeros((1, 32, D), dtype=torch.float32, device="cuda")
    with pytest.raises(TypeError):  # queries must be bf16
        pa.attention_fp8(q.clone(), q, kc, vc, torch.zeros((1, 1), dtype=torch.int32, device="cuda"),
                         torch.ones(1, dtype=torch.int32, device="cuda"),
                         torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                         max_query_len=1, max_seq_len=1, scale=0.1, k_scale=1.0, v_scale=1.0)
    with pytest.raises(pa.PAError):  # a non-positive scale is rejected before any launch
        pa.kv_write_fp8(torch.zeros((1, H, D), dtype=torch.bfloat16, device="cuda"),
                        torch.zeros((1, H, D), dtype=torch.bfloat16, device="cuda"), kc, vc,
                        torch.zeros(1, dtype=torch.int64, device="cuda"), 0.0, 1.0)


FP8_PREFILL_EDGE = [
    # (name, spec, ctx, q_lens)
    ("g4_b16_mixed", workloads.Spec("bf16", 32, 8, 128, 16, 0.088), [0, 100, 300, 7, 900], [200, 77, 5, 1, 1]),
    ("g1_b64", workloads.Spec("bf16", 8, 8, 128, 64, 0.088), [50, 0], [130, 300]),
    ("g2_b128", workloads.Spec("bf16", 8, 4, 128, 128, 0.088), [129, 0], [40, 256]),
    ("g8_b8", workloads.Spec("bf16", 32, 4, 128, 8, 0.088), [17, 0], [60, 2]),
    ("g4_b32_long_prior", workloads.Spec("bf16", 32, 8, 128, 32, 0.088), [3000], [300]),
]


@pytest.mark.parametrize("name,spec,ctx,q_lens", FP8_PREFILL_EDGE, ids=[e[0] for e in FP8_PREFILL_EDGE])
def test_fp8_prefill_edge_cases(pa, name, spec, ctx, q_lens):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    wl = workloads.with_fp8_cache(workloads.custom(spec, ctx, q_lens, name=name), k_scale=2.0 ** -5,
                                  v_scale=0.0173)
    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    dw.run_step(st)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    ref = run_workload(wl)
    assert np.array_equal(torch_to_storage(dw.k_cache), ref.k_cache)
    _close(torch_to_storage(st.out), ref.out, name)


def test_fp8_full_size_mixed_all_requests(pa):
    """The mixed batch (8 chunks of 512 queries + 248 decodes) over an E4M3 cache: every
    request's rows against the oracle."""
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    wl = workloads.with_fp8_cache(workloads.build(5))
    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    dw.run_step(st)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    ref = run_workload(wl)
    assert np.array_equal(torch_to_storage(dw.k_cache), ref.k_cache)
    _close(torch_to_storage(st.out), ref.out, wl.name)


@pytest.mark.parametrize("size,caching", [("small", True), ("small", False), ("full", True)])
def test_fp8_system_prompt(pa, size, caching):
    """Requests reusing a cached system prompt (or computing it all) over an E4M3 cache."""
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    wl = workloads.with_fp8_cache(workloads.system_prompt(size, caching=caching))
    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    dw.run_step(st)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    n = wl.meta["requests"]
    pick = list(range(n)) if size == "small" else [0, 17, 40, 63]
    ref = run_workload(wl, eval_seqs=None if size == "small" else pick)
    assert np.array_equal(st.query_start_loc.cpu().numpy(), ref.query_start_loc)
    qsl = ref.query_start_loc
    rows = np.concatenate([np.arange(qsl[i], qsl[i + 1]) for i in pick])
    _close(torch_to_storage(st.out)[rows], ref.out[rows], wl.name)
