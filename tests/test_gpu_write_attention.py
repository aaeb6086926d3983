"""pa_write_attention (the cache write fused into the attention call) vs the oracle.

The fused call must leave the same cache bytes as pa_kv_write and give the outputs the
oracle gives for write-then-attend (same bars as the unfused path), and its decode
outputs must be bit-identical to pa_kv_write + pa_attention on the same inputs.
"""
import numpy as np
import pytest
import torch

import workloads
from errmodel import assert_close_bf16, batch_sigma
from oracle import paged_attention_ref, run_workload, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_161_gb300 as m

    m.read_device_errors(clear=True)
    return m


def _close(got, ref, dtype, what, res=None, spec=None):
    """Pass bar; with the oracle result ``res`` (bf16) also the diagnostic bound of
    tests/errmodel.py over all of its rows."""
    err = np.abs(to_f64(got) - ref)
    if dtype == "f32":
        assert np.max(err) <= 2e-5, f"{what}: max err {np.max(err)}"
    elif res is not None:
        sig = batch_sigma(res, range(len(res.seq_lens)), spec.scale, spec.block_size)
        assert_close_bf16(to_f64(got), ref, sig, what)
    else:
        bad = err > 1.5e-2 + 1e-2 * np.abs(ref)
        assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance"


def _fused_step(pa, wl, eval_seqs=None):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload, torch_to_storage

    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    assert dw.fusable(st)
    dw.run_step(st, fused=True)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    return dw, st, torch_to_storage(st.out), run_workload(wl, eval_seqs=eval_seqs), torch_to_storage


@pytest.mark.parametrize("cfg", [1, 3, 4, 5])
def test_fused_small_workload_matches_oracle(pa, cfg):
    wl = workloads.build(cfg, "small")
    dw, st, out, ref, t2s = _fused_step(pa, wl)
    assert np.array_equal(t2s(dw.k_cache), ref.k_cache)
    assert np.array_equal(t2s(dw.v_cache), ref.v_cache)
    _close(out, ref.out, wl.spec.dtype, wl.name, ref, wl.spec)


def test_fused_full_size_gqa_decode_batch(pa):
    """The 256-request GQA decode batch as the benchmark runs it: the new token of every
    request is in the cache, the caches equal the oracle's, and every request's output
    matches the oracle."""
    wl = workloads.build(3)
    dw, st, out, ref, t2s = _fused_step(pa, wl)
    kc, vc = t2s(dw.k_cache), t2s(dw.v_cache)
    slots = st.slot_mapping.cpu().numpy()
    B = wl.spec.block_size
    k_new, v_new = t2s(st.k_new), t2s(st.v_new)
    for t, slot in enumerate(slots):  # every request's new row, bit-exact
        assert np.array_equal(kc[slot // B, slot % B], k_new[t])
        assert np.array_equal(vc[slot // B, slot % B], v_new[t])
    assert np.array_equal(kc, ref.k_cache) and np.array_equal(vc, ref.v_cache)
    _close(out, ref.out, wl.spec.dtype, wl.name, ref, wl.spec)


@pytest.mark.parametrize("cfg", [3, 4])
def test_fused_decode_is_bit_identical_to_write_then_attend(pa, cfg):
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    outs, caches = [], []
    for fused in (False, True):
        dw = DeviceWorkload(workloads.build(cfg, "small"))
        dw.run_setup()
        st = dw.prepare_step()
        outs.append(dw.run_step(st, fused=fused).clone())
        caches.append((dw.k_cache.clone(), dw.v_cache.clone()))
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(caches[0][0], caches[1][0]) and torch.equal(caches[0][1], caches[1][1])


FUSED_EDGE = [
    ("single_token", workloads.Spec("bf16", 32, 8, 128, 16, 0.088), [0, 0, 5], [1, 1, 1]),
    ("block_boundaries", workloads.Spec("bf16", 32, 8, 128, 16, 0.088), [15, 31, 47, 16, 32], [1] * 5),
    ("fp32_b1_g1", workloads.Spec("f32", 2, 2, 64, 1, 0.125), [9, 17], [1, 1]),
    ("bf16_b8_mqa", workloads.Spec("bf16", 4, 1, 128, 8, 0.088), [23, 8, 70], [1, 1, 1]),
    ("bf16_d64_g8_b32", workloads.Spec("bf16", 16, 2, 64, 32, 0.125), [100, 5, 64], [1, 1, 1]),
    ("mha_head_groups", workloads.Spec("bf16", 32, 32, 128, 16, 0.088), [40, 300, 1], [1, 1, 1]),
    ("many_short", workloads.Spec("bf16", 32, 8, 128, 16, 0.088), list(range(0, 300)), [1] * 300),
    ("mixed_prefill", workloads.Spec("bf16", 32, 8, 128, 16, 0.088), [0, 100, 300, 7], [200, 77, 1, 1]),
    ("mixed_fp32", workloads.Spec("f32", 8, 4, 128, 16, 0.1), [33, 70, 1], [1, 1, 3]),
]


@pytest.mark.parametrize("name,spec,ctx,q_lens", FUSED_EDGE, ids=[e[0] for e in FUSED_EDGE])
def test_fused_edge_cases(pa, name, spec, ctx, q_lens):
    wl = workloads.custom(spec, ctx, q_lens, name=name)
    dw, st, out, ref, t2s = _fused_step(pa, wl)
    assert np.array_equal(t2s(dw.k_cache), ref.k_cache)
    assert np.array_equal(t2s(dw.v_cache), ref.v_cache)
    _close(out, ref.out, spec.dtype, name, ref, spec)


def _hand_batch(dev, dtype=torch.bfloat16):
    """Three decode requests of lengths 5, 20, 33 (new token included) in a 16-block pool of
    16-token blocks, GQA 32 / 8 heads, head_dim 128; returns the pieces and each request's
    slot of its last position."""
    NB, B, Hkv, Hq, D = 16, 16, 8, 32, 128
    g = torch.Generator().manual_seed(11)
    kc = torch.randn((NB, B, Hkv, D), generator=g).to(dtype).to(dev)
    vc = torch.randn((NB, B, Hkv, D), generator=g).to(dtype).to(dev)
    lens = [5, 20, 33]
    table = torch.tensor([[3, 0, 0], [7, 1, 0], [9, 12, 4]], dtype=torch.int32)
    last = [int(table[s, (L - 1) // B]) * B + (L - 1) % B for s, L in enumerate(lens)]
    q = torch.randn((3, Hq, D), generator=g).to(dtype).to(dev)
    k_new = torch.randn((3, Hkv, D), generator=g).to(dtype).to(dev)
    v_new = torch.randn((3, Hkv, D), generator=g).to(dtype).to(dev)
    return dict(kc=kc, vc=vc, q=q, k_new=k_new, v_new=v_new, table=table.to(dev),
                lens=torch.tensor(lens, dtype=torch.int32, device=dev),
                qsl=torch.tensor([0, 1, 2, 3], dtype=torch.int32, device=dev), last=last, B=B)


def _call(pa, h, slots, fused):
    out = torch.empty_like(h["q"])
    kc, vc = h["kc"].clone(), h["vc"].clone()
    sm = torch.tensor(slots, dtype=torch.int64, device=kc.device)
    kw = dict(max_query_len=1, max_seq_len=33, scale=0.088)
    if fused:
        pa.write_attention(out, h["q"], h["k_new"], h["v_new"], sm, kc, vc, h["table"], h["lens"], h["qsl"], **kw)
    else:
        pa.kv_write(h["k_new"], h["v_new"], kc, vc, sm)
        pa.attention(out, h["q"], kc, vc, h["table"], h["lens"], h["qsl"], **kw)
    torch.cuda.synchronize()
    return out, kc, vc, pa.read_device_errors(clear=True)


def test_fused_padding_token_writes_nothing(pa):
    h = _hand_batch("cuda")
    slots = [h["last"][0], -1, h["last"][2]]
    a = _call(pa, h, slots, fused=False)
    b = _call(pa, h, slots, fused=True)
    assert a[3] == 0 and b[3] == 0
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)
    B = h["B"]
    s1 = h["last"][1]
    assert torch.equal(b[1][s1 // B, s1 % B], h["kc"][s1 // B, s1 % B])  # stale row kept
    # and the outputs are the oracle's over the cache as it stands
    ref = paged_attention_ref(_st(h["q"]), _st(b[1]), _st(b[2]), h["table"].cpu().numpy(),
                              h["lens"].cpu().numpy(), h["qsl"].cpu().numpy(), 0.088, B)
    _close(_st(b[0]), ref, "bf16", "padding")


def test_fused_slot_out_of_range_is_flagged_and_skipped(pa):
    h = _hand_batch("cuda")
    NB, B = h["kc"].shape[0], h["B"]
    slots = [h["last"][0], NB * B + 3, h["last"][2]]
    out, kc, vc, flags = _call(pa, h, slots, fused=True)
    assert flags & pa.PA_DEVERR["slot_range"]
    for s in (0, 2):
        sl = h["last"][s]
        assert torch.equal(kc[sl // B, sl % B], h["k_new"][s]) and torch.equal(vc[sl // B, sl % B], h["v_new"][s])
    kref, vref = h["kc"].clone(), h["vc"].clone()
    for s in (0, 2):
        sl = h["last"][s]
        kref[sl // B, sl % B], vref[sl // B, sl % B] = h["k_new"][s], h["v_new"][s]
    assert torch.equal(kc, kref) and torch.equal(vc, vref)  # nothing else touched


def test_fused_slot_mismatch_is_flagged(pa):
    """A decode token whose slot is not its last position's slot: flagged, its row still
    written where slot_mapping says, the other requests unaffected."""
    h = _hand_batch("cuda")
    B = h["B"]
    wrong = 15 * B + 2  # block 15 belongs to no request
    slots = [h["last"][0], wrong, h["last"][2]]
    a = _call(pa, h, slots, fused=False)
    b = _call(pa, h, slots, fused=True)
    assert a[3] == 0
    assert b[3] == pa.PA_DEVERR["slot_mismatch"]
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])  # cache as pa_kv_write leaves it
    assert torch.equal(a[0][0], b[0][0]) and torch.equal(a[0][2], b[0][2])


def test_fused_rejects_bad_arguments_before_enqueuing(pa):
    h = _hand_batch("cuda")
    out = torch.empty_like(h["q"])
    sm = torch.tensor(h["last"], dtype=torch.int64, device="cuda")
    with pytest.raises(ValueError):
        pa.write_attention(out, h["q"], h["k_new"][:2], h["v_new"], sm, h["kc"], h["vc"], h["table"], h["lens"],
                           h["qsl"], max_query_len=1, max_seq_len=33, scale=0.088)
    kc = h["kc"].clone()
    with pytest.raises(pa.PAError):  # table too narrow for max_seq_len: nothing may run
        pa.write_attention(out, h["q"], h["k_new"], h["v_new"], sm, kc, h["vc"], h["table"], h["lens"],
                           h["qsl"], max_query_len=1, max_seq_len=49, scale=0.088)
    torch.cuda.synchronize()
    assert torch.equal(kc, h["kc"])


def _st(t):
    from paged_kv_cache_161_gb300.device_workload import torch_to_storage

    return torch_to_storage(t)


@pytest.mark.parametrize("cfg,fused,fp8", [(3, True, False), (5, True, False), (1, False, False), (5, False, False),
                                           (3, False, True), (5, False, True)])
def test_output_in_pinned_host_memory_is_bit_identical(pa, cfg, fused, fp8):
    """`out` may be page-locked host memory: every attention kernel (split-K decode and its
    merge, the tensor-core and CUDA-core prefill, E4M3 caches) then stores its rows over the
    CPU-GPU link, with the same bits as into device memory."""
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    wl = workloads.build(cfg, "small")
    if fp8:
        wl = workloads.with_fp8_cache(wl)
    outs = []
    for host in (False, True):
        dw = DeviceWorkload(wl)
        dw.run_setup()
        st = dw.prepare_step()
        if host:
            st.out = torch.full(st.out.shape, float("nan"), dtype=st.out.dtype).pin_memory()
        outs.append(dw.run_step(st, fused=fused))
        torch.cuda.synchronize()
        assert pa.read_device_errors(clear=True) == 0
    assert not outs[1].is_cuda
    assert torch.equal(outs[0].cpu(), outs[1])


def test_grouped_output_in_pinned_host_memory(pa):
    """The grouped decode (shared-prefix segments and their merge) into pinned host memory."""
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    wl = workloads.build(4, "small")
    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    dw.run_step(st)
    seq_group, group_range, shared_len = dw.bm.batch_groups([s for s, _ in wl.step.batch], 4)
    dev = st.q.device
    args = (st.q, dw.k_cache, dw.v_cache, st.block_table, st.seq_lens, st.query_start_loc,
            torch.from_numpy(seq_group).to(dev), torch.from_numpy(group_range).to(dev),
            torch.from_numpy(shared_len).to(dev))
    out_d = torch.empty_like(st.q)
    out_h = torch.full(st.q.shape, float("nan"), dtype=st.q.dtype).pin_memory()
    for out in (out_d, out_h):
        pa.attention_grouped(out, *args, max_seq_len=st.max_seq_len, scale=wl.spec.scale)
    torch.cuda.synchronize()
    assert pa.read_device_errors(clear=True) == 0
    assert len(group_range) > 0
    assert torch.equal(out_d.cpu(), out_h)


def test_mixed_calls_from_two_host_threads(pa):
    """Mixed decode + prefill calls fork the library's internal stream; calls issued at once
    from two host threads, on two streams with two workspaces, give the single-call bits."""
    import threading

    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    wl = workloads.build(5, "small")
    dw = DeviceWorkload(wl)
    dw.run_setup()
    st = dw.prepare_step()
    kw = dict(max_query_len=st.max_query_len, max_seq_len=st.max_seq_len, scale=wl.spec.scale)
    args = (st.q, dw.k_cache, dw.v_cache, st.block_table, st.seq_lens, st.query_start_loc)
    ref = torch.empty_like(st.q)
    pa.attention(ref, *args, workspace=st.workspace, **kw)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.full_like(st.q, float("nan")) for _ in streams]
    wss = [torch.empty_like(st.workspace) for _ in streams]
    errors = []

    def work(i):
        try:
            for _ in range(20):
                pa.attention(outs[i], *args, workspace=wss[i], stream=streams[i], **kw)
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert pa.read_device_errors(clear=True) == 0
    for out in outs:
        assert torch.equal(out, ref)


def test_decode_rows_in_pinned_host_memory(pa, monkeypatch):
    """q, k_new and v_new in pinned host memory (decode-only batch): the decode kernel reads
    them over the CPU-GPU link; the cache and the output bits equal the device-input call's.
    Pageable host memory, and host rows with a prefill row in the batch, are refused before
    anything is enqueued."""
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    outs, caches = [], []
    for host in (False, True):
        wl = workloads.build(3, "small")
        dw = DeviceWorkload(wl)
        dw.run_setup()
        st = dw.prepare_step()
        q, k, v = st.q, st.k_new, st.v_new
        if host:
            q, k, v = (t.cpu().pin_memory() for t in (q, k, v))
        out = torch.full_like(st.q, float("nan"))
        pa.write_attention(out, q, k, v, st.slot_mapping, dw.k_cache, dw.v_cache, st.block_table, st.seq_lens,
                           st.query_start_loc, max_query_len=1, max_seq_len=st.max_seq_len, scale=wl.spec.scale,
                           workspace=st.workspace)
        out2 = torch.full_like(st.q, float("nan"))
        pa.attention(out2, q, dw.k_cache, dw.v_cache, st.block_table, st.seq_lens, st.query_start_loc,
                     max_query_len=1, max_seq_len=st.max_seq_len, scale=wl.spec.scale, workspace=st.workspace)
        torch.cuda.synchronize()
        assert pa.read_device_errors(clear=True) == 0
        assert torch.equal(out, out2)
        outs.append(out)
        caches.append((dw.k_cache.clone(), dw.v_cache.clone()))
        if host:
            # the library's own check (past the binding's): pageable host memory is refused
            monkeypatch.setattr(pa, "_pool_ptr", lambda t, name: t.data_ptr())
            with pytest.raises(pa.PAError):
                pa.attention(torch.empty_like(st.q), st.q.cpu(), dw.k_cache, dw.v_cache, st.block_table,
                             st.seq_lens, st.query_start_loc, max_query_len=1, max_seq_len=st.max_seq_len,
                             scale=wl.spec.scale, workspace=st.workspace)
            with pytest.raises(pa.PAError):  # host rows with max_query_len >= 2: refused
                pa.attention(torch.empty_like(st.q), q, dw.k_cache, dw.v_cache, st.block_table, st.seq_lens,
                             st.query_start_loc, max_query_len=2, max_seq_len=st.max_seq_len,
                             scale=wl.spec.scale, workspace=st.workspace)
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(caches[0][0], caches[1][0]) and torch.equal(caches[0][1], caches[1][1])
