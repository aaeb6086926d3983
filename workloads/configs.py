"""The five paged-attention workloads, full size and reduced, plus a custom builder.

A workload is a pool of physical blocks, the order in which free block ids are
handed out, and a script of phases. A phase is a list of block-manager
operations followed, optionally, by one attention batch:

    ('add', s)            start an empty sequence s
    ('append', s, n)      append n new tokens to s (their K/V are then written)
    ('fork', p, c)        c starts as a copy of p's block table (shared blocks)
    ('prompt', s, n)      admit s with the first n tokens of its token stream: with
                          prefix caching, start from whatever prefix the block manager
                          can reuse, then append the rest; without, append all n
    ('free', s)           the request s ends
    ('fill', s)           append to the empty sequence s as many tokens as the free
                          blocks hold (num_free * block_size, from the block manager)
    ('swap_out', seqs)    preempt the group ``seqs`` (a tuple): its blocks go to the CPU
    ('swap_in', seqs)     bring the group back to the GPU

Swap operations sit in phases without appends; their block copies run after the
phase's copy-on-write copies, in operation order.

A batch entry (s, None) means "the tokens appended to s in this phase" (the count a
'prompt' op leaves depends on what the block manager reused). Workloads with
``token_ids`` give every sequence a stream of token ids; ``shared_kv`` maps a sequence
to (owner, n): its first n positions hold the owner's K/V (the same tokens at the same
positions give the same K/V), and ``q_whole`` makes a sequence's queries slices of one
draw over its whole length, so rows at the same position agree however they are batched.

Both the oracle and the CUDA path execute a phase the same way: run the
operations on their own block manager, apply the copy-on-write pairs it emitted
(in emission order), write the K/V of every appended token through the slot
mapping (in operation order), then run attention over ``batch`` -- a list of
(sequence, q_len) whose query rows are the last q_len tokens of each sequence.
How slots, tables and pairs are derived is the method's business and is not
here.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 161000
# Replica r of a workload (one per rank when a benchmark runs on several GPUs) draws from
# seed + REPLICA_STRIDE * r: same shapes and distributions, its own lengths and values.
REPLICA_STRIDE = 1000
_KIND_K, _KIND_V, _KIND_Q, _KIND_STRUCT = 1, 2, 3, 0


@dataclass(frozen=True)
class Spec:
    dtype: str  # 'f32' or 'bf16': the storage and I/O type of q, K, V and out
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def kv_token_bytes(self) -> int:
        """Bytes of K plus V for one token over all KV heads."""
        return 2 * self.num_kv_heads * self.head_dim * self.elem_bytes


@dataclass
class Phase:
    ops: list = field(default_factory=list)
    batch: list | None = None


@dataclass
class Workload:
    name: str
    spec: Spec
    seed: int
    num_blocks: int
    free_order: np.ndarray  # int32 permutation of range(num_blocks)
    setup: list
    step: Phase
    num_seqs: int
    meta: dict = field(default_factory=dict)
    prefix_caching: bool = False
    token_ids: dict = field(default_factory=dict)  # seq -> int32 array (its token stream)
    shared_kv: dict = field(default_factory=dict)  # seq -> (owner, n)
    q_whole: dict = field(default_factory=dict)  # seq -> length of its one query draw
    cpu_blocks: int = 0  # CPU block pool for swapping (0: none)
    cpu_free_order: np.ndarray | None = None
    kv_cache: str = ""  # cache element type: "" (the spec's dtype) or "fp8_e4m3"
    k_scale: float = 1.0  # fp8_e4m3: a K code c stands for value(c) * k_scale
    v_scale: float = 1.0

    # ---- random values -------------------------------------------------
    def _normal(self, kind: int, seq: int, start: int, shape) -> np.ndarray:
        ss = np.random.SeedSequence([self.seed, kind, seq, start])
        x = np.random.Generator(np.random.PCG64(ss)).standard_normal(shape, dtype=np.float32)
        return _to_storage(x, self.spec.dtype)

    def _whole(self, kind: int, seq: int, n: int, width: int) -> np.ndarray:
        cache = self.__dict__.setdefault("_whole_cache", {})
        key = (kind, seq, n)
        if key not in cache:
            cache[key] = self._normal(kind, seq, 0, (n, width, self.spec.head_dim))
        return cache[key]

    def kv(self, seq: int, start: int, n: int):
        """K and V of tokens [start, start+n) of ``seq``: storage arrays [n, Hkv, D]."""
        Hkv = self.spec.num_kv_heads
        shp = (n, Hkv, self.spec.head_dim)
        own = self.shared_kv.get(seq)
        if own is None or start >= own[1]:
            return self._normal(_KIND_K, seq, start, shp), self._normal(_KIND_V, seq, start, shp)
        owner, ns = own
        n1 = min(n, ns - start)
        k = self._whole(_KIND_K, owner, ns, Hkv)[start:start + n1]
        v = self._whole(_KIND_V, owner, ns, Hkv)[start:start + n1]
        if n1 < n:
            k2, v2 = self.kv(seq, ns, n - n1)
            k, v = np.concatenate([k, k2]), np.concatenate([v, v2])
        return k, v

    def q(self, seq: int, start: int, n: int) -> np.ndarray:
        """Queries of tokens [start, start+n) of ``seq``: storage array [n, Hq, D]."""
        if seq in self.q_whole:
            return self._whole(_KIND_Q, seq, self.q_whole[seq], self.spec.num_heads)[start:start + n]
        return self._normal(_KIND_Q, seq, start, (n, self.spec.num_heads, self.spec.head_dim))

    def tokens(self, seq: int, start: int, n: int) -> np.ndarray:
        """Token ids of positions [start, start+n) of ``seq``."""
        return np.asarray(self.token_ids[seq][start:start + n], np.int32)

    def kv_many(self, reqs, threads: int | None = None):
        """``kv`` for a list of (seq, start, n), drawn on a thread pool."""
        threads = threads or min(16, len(os.sched_getaffinity(0)))
        if len(reqs) <= 2:
            return [self.kv(*r) for r in reqs]
        with ThreadPoolExecutor(threads) as ex:
            return list(ex.map(lambda r: self.kv(*r), reqs))

    # ---- token bookkeeping (lengths only) --------------------------------
    def phases(self):
        return list(self.setup) + [self.step]

    def step_queries(self, lens: dict | None = None, appended: dict | None = None):
        """(seq, start, q_len) of every query range of the step's batch, in batch order.

        ``lens`` (final lengths) and ``appended`` (tokens appended to each sequence in the
        step) come from a block manager when the script has 'prompt' operations."""
        if lens is None:
            lens = {}
            for ph in self.phases():
                for op in ph.ops:
                    if op[0] == "add":
                        lens[op[1]] = 0
                    elif op[0] == "append":
                        lens[op[1]] += op[2]
                    elif op[0] == "fork":
                        lens[op[2]] = lens[op[1]]
                    elif op[0] == "prompt":
                        raise ValueError("'prompt' lengths depend on the block manager: pass lens")
        out = []
        for s, ql in self.step.batch or []:
            q = appended.get(s, 0) if ql is None else ql
            out.append((s, lens[s] - q, q))
        return out

    def appends(self, phase: Phase, lens: dict):
        """(seq, start, n) of each append of ``phase``; ``lens`` is advanced in place."""
        out = []
        for op in phase.ops:
            if op[0] == "add":
                lens[op[1]] = 0
            elif op[0] == "append":
                out.append((op[1], lens[op[1]], op[2]))
                lens[op[1]] += op[2]
            elif op[0] == "fork":
                lens[op[2]] = lens[op[1]]
        return out


def _to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return x
    # float32 -> bfloat16 bit pattern, round to nearest even (inputs are finite)
    u = x.view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def relevant_seqs(wl: Workload, seqs) -> set:
    """``seqs`` together with every sequence they were forked from or share K/V with."""
    parent = {}
    for ph in wl.phases():
        for op in ph.ops:
            if op[0] == "fork":
                parent[op[2]] = op[1]
    out = set()
    todo = list(seqs)
    while todo:
        s = todo.pop()
        if s is None or s in out:
            continue
        out.add(s)
        todo.append(parent.get(s))
        if s in wl.shared_kv:
            todo.append(wl.shared_kv[s][0])
    return out


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _KIND_STRUCT])))


def _pool(needed_blocks: int, factor: float = 1.25) -> int:
    return int(math.ceil(factor * needed_blocks))


GQA = dict(num_heads=32, num_kv_heads=8, head_dim=128, block_size=16, scale=1.0 / math.sqrt(128))


# ---------------------------------------------------------------------------
def _decode_workload(name, spec, seed, ctx, write_step, rng, pool=None, meta=None):
    """Sequences with ``ctx`` cached tokens; the step appends one token each (if
    ``write_step``) and runs one decode query per sequence."""
    S = len(ctx)
    B = spec.block_size
    setup = Phase(ops=[("add", s) for s in range(S)] + [("append", s, int(L)) for s, L in enumerate(ctx) if L > 0])
    if write_step:
        step = Phase(ops=[("append", s, 1) for s in range(S)], batch=[(s, 1) for s in range(S)])
        final = [int(L) + 1 for L in ctx]
    else:
        step = Phase(ops=[], batch=[(s, 1) for s in range(S)])
        final = [int(L) for L in ctx]
    if pool is None:
        pool = _pool(sum(-(-L // B) for L in final))
    return Workload(name, spec, seed, pool, rng.permutation(pool).astype(np.int32), [setup], step, S,
                    dict(meta or {}, final_lens=final))


def _cfg1(size, replica=0):
    seed = SEED_BASE + 1 + REPLICA_STRIDE * replica
    spec = Spec("f32", 4, 4, 64, 4, 1.0 / 8)
    rng = _rng(seed)
    return _decode_workload("tiny_fp32_decode", spec, seed, [7, 16, 33], True, rng, pool=64)


def _cfg2(size, replica=0):
    seed = SEED_BASE + 2 + (100 if size == "small" else 0) + REPLICA_STRIDE * replica
    spec = Spec("bf16", 32, 32, 128, 16, 1.0 / math.sqrt(128))
    rng = _rng(seed)
    if size == "small":
        ctx = rng.integers(16, 160, size=6, endpoint=True)
    else:
        ctx = rng.integers(128, 2048, size=64, endpoint=True)
    return _decode_workload("mha_bf16_decode" + ("_small" if size == "small" else ""), spec, seed, ctx, False, rng)


def _cfg3(size, replica=0):
    seed = SEED_BASE + 3 + (100 if size == "small" else 0) + REPLICA_STRIDE * replica
    spec = Spec("bf16", **GQA)
    rng = _rng(seed)
    if size == "small":
        S, med, lo, hi = 12, 100, 1, 600
    else:
        S, med, lo, hi = 256, 1024, 16, 8192
    ctx = np.clip(np.rint(rng.lognormal(math.log(med), 1.0, size=S)), lo, hi).astype(np.int64)
    return _decode_workload("gqa_bf16_decode_b256" + ("_small" if size == "small" else ""), spec, seed, ctx,
                            True, rng, meta=dict(lognormal_sigma=1.0, median=med, clip=(lo, hi)))


def _cfg4(size, replica=0):
    seed = SEED_BASE + 4 + (100 if size == "small" else 0) + REPLICA_STRIDE * replica
    if size == "small":
        return shared_prefix(3, 40, 4, 20, seed, "shared_prefix_bf16_small")
    return shared_prefix(64, 1000, 4, 256, seed, "shared_prefix_bf16")


def shared_prefix(P: int, prompt_len: int, n_samp: int, tail_hi: int, seed: int,
                  name: str = "shared_prefix_custom") -> Workload:
    """P prompts of prompt_len tokens, n_samp samples forked from each (the prompt's blocks
    shared, the partial last block copied on write), tails U[0, tail_hi] appended to every
    sample, then one decode token per sample; GQA 32 q / 8 kv heads, head_dim 128, block 16."""
    spec = Spec("bf16", **GQA)
    rng = _rng(seed)
    B = spec.block_size
    tails = rng.integers(0, tail_hi, size=(P, n_samp), endpoint=True)
    seq = lambda p, i: p * n_samp + i  # noqa: E731
    prompt = Phase(ops=[op for p in range(P) for op in (("add", seq(p, 0)), ("append", seq(p, 0), prompt_len))])
    fork = Phase(ops=[("fork", seq(p, 0), seq(p, i)) for p in range(P) for i in range(1, n_samp)])
    tail = Phase(ops=[("append", seq(p, i), int(tails[p, i])) for p in range(P) for i in range(n_samp)
                      if tails[p, i] > 0])
    S = P * n_samp
    step = Phase(ops=[("append", s, 1) for s in range(S)], batch=[(s, 1) for s in range(S)])
    shared_full = prompt_len // B
    needed = 0
    for p in range(P):
        needed += shared_full + sum(-(-(prompt_len + int(t) + 1) // B) - shared_full for t in tails[p])
    pool = _pool(needed)
    final = [prompt_len + int(tails[p, i]) + 1 for p in range(P) for i in range(n_samp)]
    return Workload(name, spec, seed, pool, rng.permutation(pool).astype(np.int32), [prompt, fork, tail], step, S,
                    dict(prompts=P, prompt_len=prompt_len, samples=n_samp, tails=tails, final_lens=final))


def _cfg5(size, replica=0):
    seed = SEED_BASE + 5 + (100 if size == "small" else 0) + REPLICA_STRIDE * replica
    spec = Spec("bf16", **GQA)
    rng = _rng(seed)
    if size == "small":
        n_chunk, chunk, prior_hi, n_dec, dec_lo, dec_hi = 2, 200, 300, 10, 16, 300
    else:
        n_chunk, chunk, prior_hi, n_dec, dec_lo, dec_hi = 8, 512, 4096, 248, 256, 4096
    prior = rng.integers(0, prior_hi, size=n_chunk, endpoint=True)
    dec = rng.integers(dec_lo, dec_hi, size=n_dec, endpoint=True)
    S = n_chunk + n_dec
    ctx = list(prior) + list(dec)
    qlen = [chunk] * n_chunk + [1] * n_dec
    setup = Phase(ops=[("add", s) for s in range(S)] + [("append", s, int(L)) for s, L in enumerate(ctx) if L > 0])
    step = Phase(ops=[("append", s, q) for s, q in enumerate(qlen)], batch=[(s, q) for s, q in enumerate(qlen)])
    B = spec.block_size
    final = [int(L) + q for L, q in zip(ctx, qlen)]
    pool = _pool(sum(-(-L // B) for L in final))
    return Workload("mixed_prefill_decode_bf16" + ("_small" if size == "small" else ""), spec, seed, pool,
                    rng.permutation(pool).astype(np.int32), [setup], step, S,
                    dict(chunks=n_chunk, chunk_len=chunk, prior=prior, decode_ctx=dec, final_lens=final))


def with_fp8_cache(wl: Workload, k_scale: float = 2.0 ** -6, v_scale: float = 2.0 ** -6) -> Workload:
    """The same workload over an FP8 (E4M3) cache: inputs unchanged, the cache stores
    E4M3(x / scale). The default scales (2^-6) put N(0, 1) values well inside E4M3's range
    (|x| < 7 for every draw here -> codes below 448)."""
    import dataclasses

    return dataclasses.replace(wl, name=wl.name + "_fp8", kv_cache="fp8_e4m3", k_scale=float(k_scale),
                               v_scale=float(v_scale))


def preemption(size: str = "full") -> Workload:
    """Preemption by swapping (the code-reading page's SequenceGroup lifecycle): groups of 4
    samples forked from one prompt (tails written with copy-on-write); group 0 is swapped
    out to the CPU; a long request then takes every free GPU block (overwriting group 0's
    old blocks) and ends; group 0 is swapped back in; the step decodes every sample (one
    new token each). Full: 16 groups, 1000-token prompts, tails U[0, 256]. Small: 3 groups,
    40-token prompts, tails U[0, 20]."""
    seed = SEED_BASE + 7 + (100 if size == "small" else 0)
    spec = Spec("bf16", **GQA)
    rng = _rng(seed)
    if size == "small":
        P, prompt_len, n_samp, tail_hi = 3, 40, 4, 20
    else:
        P, prompt_len, n_samp, tail_hi = 16, 1000, 4, 256
    B = spec.block_size
    tails = rng.integers(0, tail_hi, size=(P, n_samp), endpoint=True)
    seq = lambda p, i: p * n_samp + i  # noqa: E731
    S = P * n_samp
    hog = S
    prompt = Phase(ops=[op for p in range(P) for op in (("add", seq(p, 0)), ("append", seq(p, 0), prompt_len))])
    fork = Phase(ops=[("fork", seq(p, 0), seq(p, i)) for p in range(P) for i in range(1, n_samp)])
    tail = Phase(ops=[("append", seq(p, i), int(tails[p, i])) for p in range(P) for i in range(n_samp)
                      if tails[p, i] > 0])
    group0 = tuple(seq(0, i) for i in range(n_samp))
    shared_full = prompt_len // B
    # pool: 1.25x an upper bound of the blocks all samples hold after the step
    per_group = [shared_full + sum(-(-(prompt_len + int(t) + 1) // B) - shared_full + 1 for t in tails[p])
                 for p in range(P)]
    pool = _pool(sum(per_group))
    swap_out = Phase(ops=[("swap_out", group0)])
    hog_phase = Phase(ops=[("add", hog), ("fill", hog)])  # overwrites group 0's old blocks
    back = Phase(ops=[("free", hog)])
    swap_in = Phase(ops=[("swap_in", group0)])
    step = Phase(ops=[("append", s, 1) for s in range(S)], batch=[(s, 1) for s in range(S)])
    cpu_blocks = int(math.ceil(1.5 * per_group[0]))
    final = [prompt_len + int(tails[p, i]) + 1 for p in range(P) for i in range(n_samp)]
    return Workload("preemption_swap_bf16" + ("_small" if size == "small" else ""), spec, seed, pool,
                    rng.permutation(pool).astype(np.int32), [prompt, fork, tail, swap_out, hog_phase, back, swap_in],
                    step, S, dict(groups=P, prompt_len=prompt_len, samples=n_samp, tails=tails, final_lens=final,
                                  swapped_group=list(group0)),
                    cpu_blocks=cpu_blocks, cpu_free_order=rng.permutation(cpu_blocks).astype(np.int32))


def system_prompt(size: str = "full", caching: bool = True) -> Workload:
    """Many requests sharing one system prompt (the prefix-caching case of the docs page).

    A warm request computes the system prompt and ends (its blocks are released, still
    cached when ``caching``). The step admits R requests, each the system prompt plus its
    own user text, as one chunked-prefill batch: with caching each request reuses the
    prompt's full blocks and computes only the rest; without, it computes everything.
    Full: R = 64, a 2040-token system prompt (127 full blocks + 8 tokens), user text
    U[64, 512] tokens. Small: R = 6, 100-token prompt, user text U[5, 40].
    """
    seed = SEED_BASE + 6 + (100 if size == "small" else 0)
    spec = Spec("bf16", **GQA)
    rng = _rng(seed)
    if size == "small":
        R, P, ulo, uhi = 6, 100, 5, 40
    else:
        R, P, ulo, uhi = 64, 2040, 64, 512
    vocab = 32000
    sys_tokens = rng.integers(0, vocab, size=P)
    user_lens = [int(u) for u in rng.integers(ulo, uhi, size=R, endpoint=True)]
    W = R  # the warm request
    token_ids = {W: sys_tokens.astype(np.int32)}
    for r in range(R):
        token_ids[r] = np.concatenate([sys_tokens, rng.integers(0, vocab, size=user_lens[r])]).astype(np.int32)
    B = spec.block_size
    pool = _pool(sum(-(-(P + u) // B) for u in user_lens))
    setup = [Phase(ops=[("prompt", W, P), ("free", W)])]
    step = Phase(ops=[("prompt", r, P + user_lens[r]) for r in range(R)], batch=[(r, None) for r in range(R)])
    name = "system_prompt_bf16_" + ("cached" if caching else "uncached") + ("_small" if size == "small" else "")
    return Workload(name, spec, seed, pool, rng.permutation(pool).astype(np.int32), setup, step, R,
                    dict(requests=R, system_len=P, user_lens=user_lens, final_lens=[P + u for u in user_lens]),
                    prefix_caching=caching, token_ids=token_ids, shared_kv={s: (W, P) for s in range(R + 1)},
                    q_whole={r: P + user_lens[r] for r in range(R)})


CONFIGS = {1: _cfg1, 2: _cfg2, 3: _cfg3, 4: _cfg4, 5: _cfg5}


def build(config: int, size: str = "full", replica: int = 0) -> Workload:
    """Workload ``config`` (1..5) at ``size`` 'full' or 'small'; ``replica`` r > 0 gives an
    independent draw of the same workload (seed + REPLICA_STRIDE * r)."""
    if size not in ("full", "small"):
        raise ValueError(size)
    if replica < 0:
        raise ValueError(replica)
    return CONFIGS[config](size, replica)


def custom(spec: Spec, ctx, q_lens, seed: int = SEED_BASE + 999, pool: int | None = None,
           pool_factor: float = 1.25, name: str = "custom") -> Workload:
    """Sequences with ``ctx[s]`` cached tokens; the step appends ``q_lens[s]``
    tokens to each and attends with those as queries (q_len 0 = no query rows)."""
    S = len(ctx)
    B = spec.block_size
    rng = _rng(seed)
    setup = Phase(ops=[("add", s) for s in range(S)] + [("append", s, int(L)) for s, L in enumerate(ctx) if L > 0])
    step = Phase(ops=[("append", s, int(q)) for s, q in enumerate(q_lens) if q > 0],
                 batch=[(s, int(q)) for s, q in enumerate(q_lens)])
    final = [int(L) + int(q) for L, q in zip(ctx, q_lens)]
    if pool is None:
        pool = max(1, _pool(sum(-(-L // B) for L in final), pool_factor))
    return Workload(name, spec, seed, pool, rng.permutation(pool).astype(np.int32), [setup], step, S,
                    dict(final_lens=final))
