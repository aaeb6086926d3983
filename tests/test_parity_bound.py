"""The diagnostic bound of tests/errmodel.py, on the CPU.

1. Calibration: a CPU model of the kernels' rounding (bf16 inputs, fp32 logits and sums,
   16-key stages with a running maximum, bf16 softmax numerators, one bf16 rounding of
   the result) stays inside the bound with margin at every context length.
2. Mutations: the float64 oracle's output for the longest request of the GQA batch-256
   workload (and for a chunked-prefill request of the mixed workload), with keys left out
   the way a faulty kernel would leave them out -- one physical block, the request's last
   16-token stage, one 128-key prefill step of one KV head, one CTA's range of the
   split-K partition -- fails the bound, while the unmutated output rounded to bf16 and
   the rounding model pass it. At these lengths the pass bar alone does not
   see the dropped block, which is why the GPU parity tests assert both.

The oracle is the reference throughout; the mutants and the rounding model are test-side
models of kernels, not expected values.
"""
import numpy as np
import pytest

import workloads
from errmodel import U_BF16, diag_failures, northstar_failures, row_sigma
from oracle import gather_kv, run_workload, to_f64


def _bf16(x):
    """float -> nearest-even bf16, as float64."""
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def _kernel_model(q, K, V, scale, positions, lazy=False):
    """The kernels' rounding: fp32 logits (exp2 domain), 16-key stages with a running max,
    numerators rounded to bf16 for P.V, fp32 row sums of the unrounded numerators and fp32
    accumulation, result rounded to bf16. ``lazy``: the reference max moves only when a
    stage's max exceeds it by more than 8 (log2 units), so numerators reach 2^8."""
    n, Hq, D = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.zeros((n, Hq, D))
    c = np.float32(scale * 1.4426950408889634)
    for h in range(Hq):
        kh = K[:, h // G, :].astype(np.float32)
        vh = V[:, h // G, :].astype(np.float32)
        for j in range(n):
            last = int(positions[j]) + 1
            lg = (c * (kh[:last] @ q[j, h].astype(np.float32))).astype(np.float32)
            m, l, o = np.float32(-np.inf), np.float32(0), np.zeros(D, np.float32)
            for s0 in range(0, last, 16):
                sl = lg[s0:s0 + 16]
                mn = (sl.max() if sl.max() > m + 8 else m) if lazy else max(m, sl.max())
                a = np.float32(np.exp2(np.float32(m - mn)))
                p = np.exp2(sl - mn).astype(np.float32)
                l = np.float32(l * a + p.sum(dtype=np.float32))
                o = (o * a + _bf16(p).astype(np.float32) @ vh[s0:s0 + 16]).astype(np.float32)
                m = mn
            out[j, h] = _bf16(o / l)
    return out


def _masked_ref(q, K, V, scale, positions, drop):
    """float64 attention with the keys drop[key, kv_head] == True left out."""
    n, Hq, D = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.zeros((n, Hq, D))
    for h in range(Hq):
        g = h // G
        for j in range(n):
            last = int(positions[j]) + 1
            keep = ~drop[:last, g]
            lg = scale * (K[:last, g][keep] @ q[j, h])
            w = np.exp(lg - lg.max())
            out[j, h] = (w / w.sum()) @ V[:last, g][keep]
    return out


@pytest.mark.parametrize("L", [1, 2, 17, 200, 1000, 4096, 8192])
def test_rounding_model_inside_the_bound(L):
    rng = np.random.default_rng(L)
    Hq, Hkv, D = 8, 2, 128
    q = _bf16(rng.standard_normal((1, Hq, D)))
    K = _bf16(rng.standard_normal((L, Hkv, D)))
    V = _bf16(rng.standard_normal((L, Hkv, D)))
    scale = D ** -0.5
    pos = [L - 1]
    ref = _masked_ref(q, K, V, scale, pos, np.zeros((L, Hkv), bool))
    sig = row_sigma(q, K, V, scale, pos)
    got = _kernel_model(q, K, V, scale, pos)
    assert not northstar_failures(got, ref).any()
    assert not diag_failures(got, ref, sig).any()
    # the margin: the model's errors stay under half of the bound's C u sigma term
    assert not diag_failures(got, ref, sig, c=2.0).any()
    assert not diag_failures(_bf16(ref), ref, sig).any()


@pytest.mark.parametrize("L,scale", [(200, 128 ** -0.5), (4096, 128 ** -0.5), (1000, 1.0), (4096, 1.0)])
def test_lazy_max_rounding_inside_the_bound(L, scale):
    """The kernels move their reference max only past 2^8 (numerators up to 2^8 before the
    bf16 rounding); the bound holds for that arithmetic too, also for a sharp softmax
    (scale 1: logits with a standard deviation of ~11, the max moving deep into the row)."""
    rng = np.random.default_rng(L + int(scale * 1000))
    Hq, Hkv, D = 8, 2, 128
    q = _bf16(rng.standard_normal((1, Hq, D)))
    K = _bf16(rng.standard_normal((L, Hkv, D)))
    V = _bf16(rng.standard_normal((L, Hkv, D)))
    pos = [L - 1]
    ref = _masked_ref(q, K, V, scale, pos, np.zeros((L, Hkv), bool))
    sig = row_sigma(q, K, V, scale, pos)
    got = _kernel_model(q, K, V, scale, pos, lazy=True)
    assert not northstar_failures(got, ref).any()
    assert not diag_failures(got, ref, sig).any()


def _request(wl, i, res):
    sp = wl.spec
    a, b = int(res.query_start_loc[i]), int(res.query_start_loc[i + 1])
    L = int(res.seq_lens[i])
    K = gather_kv(res.k_cache, res.block_table[i], L, sp.block_size)
    V = gather_kv(res.v_cache, res.block_table[i], L, sp.block_size)
    return to_f64(res.q[a:b]), K, V, [L - (b - a) + j for j in range(b - a)], res.out[a:b]


@pytest.fixture(scope="module")
def gqa_longest():
    wl = workloads.build(3)
    lens = wl.meta["final_lens"]
    i = int(np.argmax(lens))
    res = run_workload(wl, eval_seqs=[i])
    return wl, _request(wl, i, res)


def _caught(wl, req, drop):
    q, K, V, pos, ref = req
    sig = row_sigma(q, K, V, wl.spec.scale, pos)
    mut = _bf16(_masked_ref(q, K, V, wl.spec.scale, pos, drop))
    return diag_failures(mut, ref, sig), northstar_failures(mut, ref)


def test_unmutated_longest_request_passes(gqa_longest):
    wl, (q, K, V, pos, ref) = gqa_longest
    assert K.shape[0] >= 8000  # the lognormal batch reaches the clip at 8192
    sig = row_sigma(q, K, V, wl.spec.scale, pos)
    assert not diag_failures(_bf16(ref), ref, sig).any()
    assert not diag_failures(_kernel_model(q, K, V, wl.spec.scale, pos), ref, sig).any()


def test_dropped_block_is_caught(gqa_longest):
    wl, req = gqa_longest
    L, Hkv = req[1].shape[0], req[1].shape[1]
    for b in (0, L // 32, (L - 1) // 16 - 1):  # first, a middle and the last full block
        drop = np.zeros((L, Hkv), bool)
        drop[16 * b:16 * b + 16] = True
        diag, ns = _caught(wl, req, drop)
        assert diag.mean() > 0.2, (b, diag.mean())
        assert ns.mean() < 0.01  # the pass bar alone (nearly) misses it at this length


def test_dropped_tail_stage_is_caught(gqa_longest):
    wl, req = gqa_longest
    L, Hkv = req[1].shape[0], req[1].shape[1]
    drop = np.zeros((L, Hkv), bool)
    drop[(L - 1) // 16 * 16:] = True  # the last stage: the partial block with the new token
    diag, _ = _caught(wl, req, drop)
    assert (L - 1) % 16 == 0  # here that stage holds the new token alone
    assert diag.sum() >= 50


def test_dropped_cta_range_is_caught(gqa_longest):
    wl, req = gqa_longest
    L, Hkv = req[1].shape[0], req[1].shape[1]
    units = sum(-(-n // 16) for n in wl.meta["final_lens"])  # 16-token stages of the batch
    span = 16 * (units // 152)  # one CTA's share on 152 SMs, in positions
    drop = np.zeros((L, Hkv), bool)
    drop[L // 3:L // 3 + span] = True
    diag, _ = _caught(wl, req, drop)
    assert diag.mean() > 0.5


def test_dropped_prefill_step_is_caught():
    wl = workloads.build(5)
    qlens = [q for _, q in wl.step.batch]
    chunks = [i for i, q in enumerate(qlens) if q > 1]
    lens = wl.meta["final_lens"]
    i = max(chunks, key=lambda c: lens[c])
    res = run_workload(wl, eval_seqs=[i])
    q, K, V, pos, ref = _request(wl, i, res)
    rows = slice(len(pos) - 32, len(pos))  # the chunk's last 32 queries (one query tile at G = 4)
    q, pos, ref = q[rows], pos[rows], ref[rows]
    L, Hkv = K.shape[0], K.shape[1]
    drop = np.zeros((L, Hkv), bool)
    drop[1024:1152, 3] = True  # one 128-key step of KV head 3
    diag, _ = _caught(wl, (q, K, V, pos, ref), drop)
    G = wl.spec.num_heads // Hkv
    hit = diag[:, 3 * G:4 * G]
    assert hit.mean() > 0.2
    assert not diag[:, :3 * G].any() and not diag[:, 4 * G:].any()  # other heads untouched
