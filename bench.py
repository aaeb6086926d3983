#!/usr/bin/env python3
"""Benchmark of the paged-KV-cache hot path on the GQA decode batch.

Workload: 256 requests, 32 query / 8 KV heads, head_dim 128, block size 16, bf16, context
lengths lognormal (median 1024, sigma 1, clipped to [16, 8192]), physical blocks handed
out in a seeded random order from a pool 1.25x the blocks needed. One step = one KV write
of the new token of every request plus one paged decode attention over all of them.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line. `value` is K/V bytes read by attention per second over the whole
step (device-resident inputs); `e2e` is the same metric through the public API with host
buffers (host block accounting, host->device copies of the step's inputs, the kernels,
device->host copy of the output waited for before the next step, all inside the timed
region; the next step's accounting overlaps the GPU's work). With --gpus N > 1 (under
torchrun) every rank runs its own batch of 256 requests (weak scaling, no collective on
the data path); `value` is all ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention: K/V GB/s (% of GB300 HBM peak) and tokens/s, batch 256"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one pa_write_attention decode
# call on this workload -- tensor-core split-K kernel (KV write fused in) plus merge kernel --
# from one ncu capture (the first timed step's two launches) of
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum \
#       --clock-control none --csv --log-file launches.csv \
#       python bench.py --steps 2 --warmup 3 --no-cpu-baseline --no-e2e --no-secondary
# It holds only for the kernel sources it was measured on (their SHA-256 below); any
# change to them makes the reported traffic null until it is measured again.
DECODE_TRAFFIC = {"sources_sha256": "e29717f03a8df0cfaa62284ccd1132765bfba070981a6dbeeb0bdddb150e47e8", "bytes": 1653156096}
DECODE_SOURCES = ["paged_kv_cache_161_gb300/csrc/decode_attention.cu", "paged_kv_cache_161_gb300/csrc/decode_mma.cu",
                  "paged_kv_cache_161_gb300/csrc/decode_common.cuh", "paged_kv_cache_161_gb300/csrc/common.cuh"]


def _decode_traffic():
    import hashlib

    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return DECODE_TRAFFIC["bytes"] if h.hexdigest() == DECODE_TRAFFIC["sources_sha256"] else None
FALLBACK_HBM_GBS = 6800.0
# End-to-end loops append one real token per request and step: two loops (rows read from
# host memory, rows copied) of at most 8 warm-up + 2 graph-check + 64 timed steps.
E2E_STEPS, E2E_WARMUP = 64, 8
E2E_TABLE_WIDTH = (8192 + 1 + 2 * (E2E_STEPS + E2E_WARMUP + 2) + 15) // 16
CONFIG_ID = 3


def _args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="leave out the other workloads' summary lines from the default run")
    ap.add_argument("--fp8", action="store_true", help="mixed / system_prompt workloads over an E4M3 cache")
    ap.add_argument("--workload", choices=["gqa_decode", "mixed", "prefill", "mha_decode", "shared_prefix",
                                           "system_prompt", "gqa_decode_fp8", "swap"],
                    default="gqa_decode",
                    help="gqa_decode: the headline line (default); mixed: the chunked-prefill + decode "
                         "batch, timed whole and as its prefill-only and decode-only sub-batches; "
                         "mha_decode: 64 requests, 32/32 heads; shared_prefix: 64 prompts x 4 samples with "
                         "copy-on-write block copies")
    a = ap.parse_args(argv)
    a.warmup = max(3, a.warmup)
    return a


def _workload_config(wl, l2_note):
    lens = [n for n in wl.meta["final_lens"]]
    sp = wl.spec
    return {
        "workload": "gqa_bf16_decode_b256: 256 requests, 32 q / 8 kv heads, head_dim 128, block 16, "
                    "lognormal context (median 1024, sigma 1, clip [16, 8192]), random block placement, "
                    "1 KV write + 1 decode attention per request",
        "global_batch": len(lens),
        "num_heads": sp.num_heads, "num_kv_heads": sp.num_kv_heads, "head_dim": sp.head_dim,
        "block_size": sp.block_size, "num_blocks": wl.num_blocks,
        "kv_tokens": int(sum(lens)), "kv_bytes_per_step": int(sum(lens)) * sp.kv_token_bytes,
        "seed": wl.seed, "l2": l2_note,
    }


# ----------------------------------------------------------------------------- multi-rank
def max_over_ranks(vals, dist=None, device="cpu"):
    """Element-wise maximum of ``vals`` over all ranks (the slowest rank's times)."""
    if dist is None:
        return [float(v) for v in vals]
    import torch

    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def sum_over_ranks(vals, dist=None, device="cpu"):
    """Element-wise sum of ``vals`` over all ranks."""
    if dist is None:
        return [float(v) for v in vals]
    import torch

    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return t.tolist()


def job_gbs(world, bytes_per_rank, ms_per_step):
    """Whole-job throughput: every rank's bytes over the slowest rank's step time."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


def rank_env():
    """(world size, rank, local rank) from the launcher's environment (1, 0, 0 without one)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_workload(rank):
    """Rank r's batch: replica r of the GQA batch-256 workload (same shapes and
    distributions, its own seed), so the ranks share nothing (weak scaling)."""
    import workloads

    return workloads.build(CONFIG_ID, replica=rank)


def _free_port():
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_command(n, argv, script=None, port=None):
    """The command that runs ``script`` (this file) as n ranks on this node, one per GPU."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr=127.0.0.1", f"--master-port={port or _free_port()}",
            script or os.path.abspath(__file__)] + list(argv)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.dev = self._smi_id(device_index)

    @staticmethod
    def _smi_id(i):
        try:
            import torch

            u = getattr(torch.cuda.get_device_properties(i), "uuid", None)
            if u is not None:
                s = str(u)
                return s if s.startswith("GPU-") else "GPU-" + s
        except Exception:
            pass
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[i] if vis else str(i)

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.dev, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- oracle timing
def _oracle_state(wl, eval_seqs):
    """Oracle caches after the untimed phases, plus the step's inputs (not timed)."""
    import numpy as np

    from oracle import BlockStore, copy_blocks_ref, kv_write_ref, run_allocator, batch_metadata
    from workloads import relevant_seqs

    sp = wl.spec
    alloc, slots_pp, copies_pp = run_allocator(wl)
    dt = np.float32 if sp.dtype == "f32" else np.uint16
    kc = BlockStore(sp.block_size, sp.num_kv_heads, sp.head_dim, dt)
    vc = BlockStore(sp.block_size, sp.num_kv_heads, sp.head_dim, dt)
    batch = wl.step.batch
    rel = relevant_seqs(wl, [batch[i][0] for i in eval_seqs])
    lens = {}
    phases = wl.phases()
    for ph, slots, copies in list(zip(phases, slots_pp, copies_pp))[:-1]:
        apps = wl.appends(ph, lens)
        copy_blocks_ref(kc, vc, copies)
        t0 = 0
        reqs = [a for a in apps if a[0] in rel]
        vals = dict(zip(reqs, wl.kv_many(reqs)))
        for a in apps:
            if a in vals:
                kv_write_ref(kc, vc, vals[a][0], vals[a][1], slots[t0:t0 + a[2]], sp.block_size)
            t0 += a[2]
    step_apps = wl.appends(wl.step, lens)
    step_vals = wl.kv_many(step_apps)
    empty = np.zeros((0, sp.num_kv_heads, sp.head_dim), np.float32 if sp.dtype == "f32" else np.uint16)
    k_new = np.concatenate([v[0] for v in step_vals]) if step_vals else empty  # (attention-only steps
    v_new = np.concatenate([v[1] for v in step_vals]) if step_vals else empty  # write nothing)
    bt, seq_lens, qsl, seqs = batch_metadata(wl, alloc)
    q = np.concatenate([wl.q(s, a, n) for s, a, n in wl.step_queries()])
    return dict(kc=kc, vc=vc, k_new=k_new, v_new=v_new, slots=slots_pp[-1], copies=copies_pp[-1], bt=bt,
                seq_lens=seq_lens, qsl=qsl, q=q)


def _oracle_step(wl, st, eval_seqs):
    """One oracle step over ``eval_seqs`` (copies, writes, attention); returns seconds."""
    from oracle import copy_blocks_ref, kv_write_ref, paged_attention_ref

    sp = wl.spec
    t = time.perf_counter()
    copy_blocks_ref(st["kc"], st["vc"], st["copies"])
    keep = set()
    for i in eval_seqs:  # the evaluated requests' new tokens
        keep.update(range(int(st["qsl"][i]), int(st["qsl"][i + 1])))
    kv_write_ref(st["kc"], st["vc"], st["k_new"], st["v_new"], st["slots"], sp.block_size, keep=keep)
    paged_attention_ref(st["q"], st["kc"], st["vc"], st["bt"], st["seq_lens"], st["qsl"], sp.scale,
                        sp.block_size, seqs=eval_seqs)
    return time.perf_counter() - t


def _cpu_sample_bytes(wl, st, eval_seqs):
    return int(sum(int(st["seq_lens"][i]) for i in eval_seqs)) * wl.spec.kv_token_bytes


def _oracle_worker(conn, replica, shard, config=CONFIG_ID):
    """One process of OraclePool: builds its shard's oracle state once (untimed), then runs
    one oracle step over the shard per request and answers with its seconds."""
    import workloads

    wl = workloads.build(config, replica=replica)
    st = _oracle_state(wl, shard) if shard else None
    conn.send(_cpu_sample_bytes(wl, st, shard) if shard else 0)
    while conn.recv():
        conn.send(_oracle_step(wl, st, shard) if shard else 0.0)
    conn.close()


class OraclePool:
    """The oracle, as it stands, over the host's cores: the step's requests ``seqs`` dealt
    round-robin to one process per core (started with spawn: this process may already hold
    a CUDA context), each holding the oracle state of its own requests. A step runs every
    shard at once; its time is the wall time until the last shard is done."""

    THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")

    def __init__(self, seqs, replica=0, workers=None, config=CONFIG_ID):
        import multiprocessing as mp

        n = workers or len(os.sched_getaffinity(0))
        self.workers = max(1, min(n, len(seqs)))
        ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        # one thread per process: the processes already cover the cores
        saved = {k: os.environ.get(k) for k in self.THREAD_VARS}
        os.environ.update({k: "1" for k in self.THREAD_VARS})
        try:
            for k in range(self.workers):
                a, b = ctx.Pipe()
                p = ctx.Process(target=_oracle_worker, args=(b, replica, list(seqs[k::self.workers]), config),
                                daemon=True)
                p.start()
                self.conns.append(a)
                self.procs.append(p)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.nbytes = sum(c.recv() for c in self.conns)  # also waits for every setup

    def step(self):
        """(wall seconds, summed per-shard CPU seconds) of one oracle step over all shards."""
        t = time.perf_counter()
        for c in self.conns:
            c.send(True)
        cpu = sum(c.recv() for c in self.conns)
        return time.perf_counter() - t, cpu

    def close(self):
        for c in self.conns:
            c.send(False)
        for p in self.procs:
            p.join(timeout=30)


def _secondary(a):
    """The other workloads at full size, summarised into the default line (one GPU): the
    mixed chunked-prefill + decode batch, MHA decode, the shared-prefix batch (plain and
    grouped decode), each with its roofline fraction and the oracle over the host's cores on
    the same workload (one whole pass: a baseline, not a target)."""
    import copy

    out = {}
    hbm, tflops, src = _peaks()
    specs = [("mixed", "mixed", 5), ("mha_decode", "mha_decode", 2), ("shared_prefix", "shared_prefix", 4)]
    for name, wname, cfg in specs:
        b = copy.copy(a)
        b.workload, b.fp8 = wname, False
        b.steps = max(30, a.steps // 4)
        try:
            ln = mixed_line(b) if name == "mixed" else secondary_line(b)
        except Exception as e:  # keep the headline line whatever happens here
            out[name] = {"error": f"{type(e).__name__}: {e}"}
            continue
        if name == "mixed":
            d = {"value": ln["value"], "unit": ln["unit"], "attention_ms": ln["attention_ms"],
                 "roofline": {"bound": "tensor", "kernel": "prefill_tc_kernel (the batch's prefill part alone)",
                              "achieved": ln["prefill"]["tflops"], "peak": tflops, "unit": "TFLOP/s",
                              "frac": ln["prefill"]["frac"], "ms": ln["prefill"]["ms"]},
                 "decode_part": {"bound": "hbm", "achieved": ln["decode"]["gbs"], "peak": hbm, "unit": "GB/s",
                                 "frac": ln["decode"]["frac"], "ms": ln["decode"]["ms"]},
                 "clocks": ln["clocks"]}
        elif name == "mha_decode":
            d = {"attention_ms": ln["attention_ms"],
                 "roofline": {"bound": "hbm", "kernel": "decode_mma_kernel + merge (pa_attention)",
                              "achieved": ln["attention_gbs_logical"], "peak": hbm, "unit": "GB/s",
                              "frac": ln["frac_logical"]}, "clocks": ln["clocks"]}
        else:
            g = ln["grouped"]
            d = {"attention_ms": ln["attention_ms"], "attention_gbs_logical": ln["attention_gbs_logical"],
                 "frac_logical": ln["attention_gbs_logical"] / hbm, "frac_unique": ln["frac_unique"],
                 "roofline": {"bound": "hbm", "kernel": "pa_attention_grouped (distinct blocks read once)",
                              "achieved": g["gbs_unique"], "peak": hbm, "unit": "GB/s", "frac": g["frac_unique"],
                              "ms": g["ms"]},
                 "copy_blocks": ln["copy_blocks"], "kv_write": ln["kv_write"], "clocks": ln["clocks"]}
        d["peak_source"] = src
        try:
            import workloads

            wl = workloads.build(cfg)
            pool = OraclePool(list(range(len(wl.step.batch))), config=cfg)
            wall, cpu = pool.step()
            pool.close()
            d["cpu_baseline"] = {"value": pool.nbytes / wall / 1e9, "unit": "GB/s of K/V", "cores": pool.workers,
                                 "kind": "oracle", "seconds": wall, "cpu_seconds": cpu,
                                 "sample": "the whole step (every request's copies, writes and attention), one pass"}
        except Exception as e:
            d["cpu_baseline"] = {"error": f"{type(e).__name__}: {e}"}
        out[name] = d
    return out


# ----------------------------------------------------------------------------- reference arm
def run_reference(a):
    import workloads

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = workloads.build(CONFIG_ID)
    sample = list(range(0, len(wl.step.batch), 8))  # 32 of the 256 requests per step
    pool = OraclePool(sample)
    for _ in range(a.warmup):
        pool.step()
    secs = [pool.step()[0] for _ in range(a.steps)]
    pool.close()
    total = sum(secs)
    nbytes = pool.nbytes
    value = nbytes * a.steps / total / 1e9
    desc = (f"{len(sample)} of the 256 requests (every 8th) per step: their copies, KV writes and attention, "
            f"dealt over {pool.workers} processes")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": a.gpus,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1e3 * total / a.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _workload_config(wl, "CPU run (no L2 rule)"),
        "tokens_per_s": len(sample) * a.steps / total,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": pool.workers, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- our arm
def run_ours(a):
    import numpy as np
    import torch

    world, rank, local = rank_env()
    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import paged_kv_cache_161_gb300 as pa
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    wl = rank_workload(rank)
    sp = wl.spec
    dw = DeviceWorkload(wl, device=dev, table_width=E2E_TABLE_WIDTH)
    dw.run_setup()
    st = dw.prepare_step()
    torch.cuda.synchronize()
    kv_bytes = int(st.seq_lens.sum().item()) * sp.kv_token_bytes
    n_req = int(st.seq_lens.shape[0])
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- device-resident timing: K steps of (KV write + attention), the write fused into
    # the decode kernel (pa_write_attention: split-K kernel + merge kernel per step)
    def fused_step():
        pa.write_attention(st.out, st.q, st.k_new, st.v_new, st.slot_mapping, dw.k_cache, dw.v_cache,
                           st.block_table, st.seq_lens, st.query_start_loc, max_query_len=st.max_query_len,
                           max_seq_len=st.max_seq_len, scale=sp.scale, workspace=st.workspace, stream=stream)

    def unfused_write():
        pa.kv_write(st.k_new, st.v_new, dw.k_cache, dw.v_cache, st.slot_mapping, stream=stream)

    def unfused_attention():
        pa.attention(st.out, st.q, dw.k_cache, dw.v_cache, st.block_table, st.seq_lens, st.query_start_loc,
                     max_query_len=st.max_query_len, max_seq_len=st.max_seq_len, scale=sp.scale,
                     workspace=st.workspace, stream=stream)

    for _ in range(a.warmup):
        fused_step()
    pa.read_device_errors(clear=True)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index)
    barrier()
    clocks.start()
    time.sleep(0.3)  # let the sampler take its first reading
    t_start.record(stream)
    for i in range(a.steps):
        ev[i][0].record(stream)
        fused_step()
        ev[i][1].record(stream)
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    flags = pa.read_device_errors(clear=True)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x}")
    step_ms = t_start.elapsed_time(t_end) / a.steps
    attn_ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / a.steps
    step_ms, attn_ms = max_over_ranks([step_ms, attn_ms], dist, dev)
    job_bytes = sum_over_ranks([kv_bytes], dist, dev)[0]  # every rank's own batch
    value = job_bytes / (step_ms * 1e-3) / 1e9

    # ---- the same step as two calls (pa_kv_write, then pa_attention), for comparison
    for _ in range(a.warmup):
        unfused_write()
        unfused_attention()
    uev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    barrier()
    t_start.record(stream)
    for i in range(a.steps):
        unfused_write()
        uev[i][0].record(stream)
        unfused_attention()
        uev[i][1].record(stream)
    t_end.record(stream)
    barrier()
    if pa.read_device_errors(clear=True):
        raise RuntimeError("device error flags set during the two-call comparison")
    u_step_ms = t_start.elapsed_time(t_end) / a.steps
    u_attn_ms = sum(e0.elapsed_time(e1) for e0, e1 in uev) / a.steps
    u_step_ms, u_attn_ms = max_over_ranks([u_step_ms, u_attn_ms], dist, dev)

    # ---- end to end through the public API with host buffers
    e2e = None
    if not a.no_e2e:
        e2e = _e2e(a, pa, dw, st, wl, dev, stream, world, dist)
        e2e_copy = _e2e(a, pa, dw, st, wl, dev, stream, world, dist, copy_rows=True)
        e2e["rows_copied_variant"] = {k: e2e_copy[k] for k in ("value", "ms_per_step", "h2d_copied_bytes_per_step")}

    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        peak, peak_src = json.load(open(peaks_path))["hbm_gbs"], "measured (MEASURED_PEAKS.json hbm_gbs)"
    else:
        peak, peak_src = FALLBACK_HBM_GBS, "fallback"
    achieved = kv_bytes / (attn_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": _decode_traffic(), "algorithmic_bytes": kv_bytes,
                "kernel": "pa_write_attention decode (tensor-core split-K kernel with the KV write fused in + merge kernel)",
                "peak_source": peak_src, "attention_ms": attn_ms,
                "frac_of_nominal_8TBs": achieved / 8000.0}

    cpu = None
    if rank == 0 and not a.no_cpu_baseline and world == 1:
        pool = OraclePool(list(range(n_req)))
        walls, cpus = [], []  # whole passes of the step (idempotent) until ~10 s of CPU work
        while sum(cpus) < 10.0 and len(walls) < 10:
            w, c = pool.step()
            walls.append(w)
            cpus.append(c)
        pool.close()
        secs = sum(walls) / len(walls)
        cpu = {"value": pool.nbytes / secs / 1e9, "unit": "GB/s", "cores": pool.workers,
               "kind": "oracle", "seconds": secs, "passes": len(walls), "cpu_seconds": sum(cpus),
               "sample": f"the whole step (all 256 requests: their KV writes and attention) dealt over "
                         f"{pool.workers} processes, {len(walls)} passes, mean wall time per pass"}

    secondary = None
    if rank == 0 and world == 1 and not a.no_secondary:
        secondary = _secondary(a)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(_workload_config(wl, f"inputs ({kv_bytes / 1e9:.2f} GB of K/V per step) larger than "
                                                 "the 129 MB L2; no flush"),
                           parallelism=f"replicas x{world} (rank r: its own batch, seed + 1000 r; no collective)"),
            "tokens_per_s": world * n_req / (step_ms * 1e-3),
            "hbm_frac_of_measured": value / (world * peak),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": a.steps * 2, "clocks": clk,
            "two_call_step": {"ms_per_step": u_step_ms, "attention_ms": u_attn_ms,
                              "value": job_bytes / (u_step_ms * 1e-3) / 1e9, "unit": "GB/s",
                              "calls": "pa_kv_write then pa_attention (3 launches), timed after the fused steps"},
        }
        if secondary is not None:
            line["secondary_workloads"] = secondary
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def _e2e(a, pa, dw, st, wl, dev, stream, world, dist, copy_rows=False):
    """Decode steps as a serving loop runs them: host block accounting (C++, one batched
    append and one table fill per step) into a pinned staging buffer, one host->device copy
    of the step's metadata (slots, tables, lengths, query_start_loc), write + attention with
    q / k / v and `out` in pinned host memory (the decode kernel reads the rows and stores
    the results over the CPU-GPU link itself; with ``copy_rows`` the rows are copied to the
    device at the start of the step instead), the result waited for before the next step is
    launched; host wall time per step. The metadata of step n + 1 does not depend on step
    n's output (one token per request), so its accounting and its copy (on a side stream,
    into the other of two device buffers) run while the GPU works on step n; the rows do
    depend on it in a serving loop, and are not fetched ahead."""
    import numpy as np
    import torch

    sp = wl.spec
    seqs = np.asarray([s for s, _ in wl.step.batch], np.int64)
    ones = np.ones(len(seqs), np.int64)
    S = len(seqs)
    width = int(st.block_table.shape[1])
    # pinned buffers holding every input of a step (two, used in turn), and one device twin;
    # the metadata first, so that its copy is one contiguous prefix
    parts = [("slots", S * 8), ("table", S * width * 4), ("lens", S * 4), ("qsl", (S + 1) * 4),
             ("q", st.q.numel() * 2), ("k", st.k_new.numel() * 2), ("v", st.v_new.numel() * 2)]
    off, offs = 0, {}
    for name, nbytes in parts:
        offs[name] = (off, nbytes)
        off += (nbytes + 255) // 256 * 256
    h_bufs = [torch.empty(off, dtype=torch.uint8).pin_memory() for _ in range(2)]
    d_bufs = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]

    def view(buf, name, dtype, shape):
        o, nb = offs[name]
        return buf[o:o + nb].view(dtype).view(shape)

    for h_buf in h_bufs:
        view(h_buf, "q", torch.bfloat16, st.q.shape).copy_(st.q.cpu())
        view(h_buf, "k", torch.bfloat16, st.k_new.shape).copy_(st.k_new.cpu())
        view(h_buf, "v", torch.bfloat16, st.v_new.shape).copy_(st.v_new.cpu())
        view(h_buf, "qsl", torch.int32, (S + 1,)).copy_(torch.arange(S + 1, dtype=torch.int32))
    host = [(view(h, "slots", torch.int64, (S,)).numpy(), view(h, "table", torch.int32, (S, width)).numpy(),
             view(h, "lens", torch.int32, (S,)).numpy()) for h in h_bufs]
    meta = offs["q"][0]  # bytes of the metadata prefix
    rows = [tuple(view(buf, n, torch.bfloat16, t.shape) for n, t in (("q", st.q), ("k", st.k_new), ("v", st.v_new)))
            for buf in (d_bufs if copy_rows else h_bufs)]
    meta_d = [(view(d, "slots", torch.int64, (S,)), view(d, "table", torch.int32, (S, width)),
               view(d, "lens", torch.int32, (S,)), view(d, "qsl", torch.int32, (S + 1,))) for d in d_bufs]
    copy_stream = torch.cuda.Stream(device=dev)
    meta_ready = [torch.cuda.Event() for _ in range(2)]
    out_h = torch.empty_like(st.q, device="cpu").pin_memory()  # written by the kernels themselves
    h2d = off
    d2h = out_h.numel() * out_h.element_size()
    bm = dw.bm
    done = torch.cuda.Event()

    def account(b):  # the next step's slots, tables and lengths into staging buffer b
        slots_h, table_h, lens_h = host[b]
        bm.append_batch(seqs, ones, out=slots_h)
        bm.batch_tables(seqs, width, table_out=table_h, lens_out=lens_h)
        return int(lens_h.max()), int(lens_h.astype(np.int64).sum()) * sp.kv_token_bytes

    def fetch_meta(b):  # staging buffer b's metadata to device buffer b, on the side stream
        with torch.cuda.stream(copy_stream):
            d_bufs[b][:meta].copy_(h_bufs[b][:meta], non_blocking=True)
            meta_ready[b].record(copy_stream)

    def enqueue(b, max_len, s):  # the step's row copy (copy_rows) and call on stream s
        if copy_rows:
            d_bufs[b][meta:].copy_(h_bufs[b][meta:], non_blocking=True)
        q_x, k_x, v_x = rows[b]
        slots_d, table_d, lens_d, qsl_d = meta_d[b]
        pa.write_attention(out_h, q_x, k_x, v_x, slots_d, dw.k_cache, dw.v_cache, table_d, lens_d, qsl_d,
                           max_query_len=1, max_seq_len=max_len, scale=sp.scale, workspace=st.workspace, stream=s)

    graphs = None  # after the warm-up: one CUDA graph per buffer pair (row copy, call)

    def run(n):
        """n steps; returns the K/V bytes of each. Buffer pair b (staging and device) is
        refilled only after the step that used it has completed (its result was waited
        for)."""
        kv = []
        nxt = account(0)
        fetch_meta(0)
        for i in range(n):
            b = i % 2
            max_len, kv_bytes = nxt
            with torch.cuda.stream(stream):
                stream.wait_event(meta_ready[b])
                if graphs is not None:
                    graphs[b].replay()
                else:
                    enqueue(b, max_len, stream)
                done.record(stream)
            if i + 1 < n:
                nxt = account(1 - b)  # overlaps the GPU's step i
                fetch_meta(1 - b)
            done.synchronize()  # step i's output is on the host
            kv.append(kv_bytes)
        return kv

    # each end-to-end step appends a real token to every request: cap the count so the
    # requests stay inside the workload's block pool (1.25x the blocks of the batch)
    steps, warm = min(a.steps, E2E_STEPS), min(a.warmup, E2E_WARMUP)
    run(warm)
    # Capture the launch side as a serving loop would (the table capacity as max_seq_len:
    # it only bounds the lengths the kernels read from the device).
    graph_note = ("CUDA graph per buffer pair (" + ("row H2D copy, " if copy_rows else "") +
                  "pa_write_attention), replayed each step after the side stream's metadata copy")
    try:
        torch.cuda.synchronize()
        captured = []
        for b in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                enqueue(b, width * sp.block_size, torch.cuda.current_stream())
            captured.append(g)
        graphs = captured
        run(2)
    except Exception as e:  # report and time the launches without a graph
        graphs = None
        graph_note = f"no CUDA graph ({type(e).__name__}: {e}); launches issued per step"
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kv_bytes_steps = run(steps)
    secs = (time.perf_counter() - t0) / steps
    secs = max_over_ranks([secs], dist, dev)[0]
    if pa.read_device_errors(clear=True):
        raise RuntimeError("device error flags set during the end-to-end run")
    mean_bytes = sum_over_ranks([sum(kv_bytes_steps) / len(kv_bytes_steps)], dist, dev)[0]
    return {"value": mean_bytes / secs / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": secs * 1e3, "steps": steps, "warmup": warm,
            "h2d_copied_bytes_per_step": off if copy_rows else meta,
            "includes": "host block accounting (pa_bm_append_batch, pa_bm_batch_tables) into pinned memory and "
                        "one H2D copy of slots/table/lens/query_start_loc, both for step n + 1 while the GPU works "
                        "on step n (two staging and two device buffers; the copy on a side stream)" +
                        ("; one H2D copy of q/k/v at the start of the step" if copy_rows else
                         "; q/k/v read by the decode kernel straight from pinned host memory (the rest of the "
                         "H2D bytes)") +
                        "; pa_write_attention storing out straight into pinned host memory (the D2H bytes), "
                        "waited for before the next step is launched",
            "launch": graph_note}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        pk = json.load(open(path))
        return pk["hbm_gbs"], pk["bf16_tflops"], "measured (MEASURED_PEAKS.json)"
    return FALLBACK_HBM_GBS, 1900.0, "fallback"


def _sub_batch(st, rows_of, idx, dev):
    """Requests `idx` of a step's batch as a batch of their own (device tensors)."""
    import torch

    qsl = st.query_start_loc.cpu()
    sel_rows = torch.cat([torch.arange(int(qsl[i]), int(qsl[i + 1])) for i in idx]).to(dev)
    q = st.q.index_select(0, sel_rows).contiguous()
    lens_q = torch.tensor([int(qsl[i + 1] - qsl[i]) for i in idx])
    new_qsl = torch.zeros(len(idx) + 1, dtype=torch.int32)
    new_qsl[1:] = torch.cumsum(lens_q, 0)
    idx_t = torch.tensor(idx, device=dev)
    return dict(q=q, out=torch.empty_like(q), block_table=st.block_table.index_select(0, idx_t).contiguous(),
                seq_lens=st.seq_lens.index_select(0, idx_t).contiguous(), query_start_loc=new_qsl.to(dev),
                max_query_len=int(lens_q.max()), max_seq_len=int(st.seq_lens.index_select(0, idx_t).max()))


def mixed_line(a):
    """The mixed chunked-prefill + decode batch (8 chunks of 512 queries with prior context
    U[0, 4096] + 248 decodes with L ~ U[256, 4096]): whole step, and each part alone."""
    import torch

    import paged_kv_cache_161_gb300 as pa
    import workloads
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    wl = workloads.build(5)
    if a.fp8:
        wl = workloads.with_fp8_cache(wl)
    sp = wl.spec
    dw = DeviceWorkload(wl, device=dev)
    dw.run_setup()
    st = dw.prepare_step()
    stream = torch.cuda.current_stream(dev)
    C = wl.meta["chunks"]
    lens = st.seq_lens.cpu().tolist()
    qlens = torch.diff(st.query_start_loc.cpu()).tolist()
    # algorithmic work: prefill flops (4 * D per query-key pair per query head), decode K/V bytes
    pf_flops = sum(4.0 * sp.head_dim * sp.num_heads * sum(lens[i] - qlens[i] + j + 1 for j in range(qlens[i]))
                   for i in range(C))
    tok_bytes = sp.kv_token_bytes // 2 if a.fp8 else sp.kv_token_bytes  # E4M3: one byte an element
    dec_bytes = sum(lens[i] for i in range(C, len(lens))) * tok_bytes
    pf_kv_bytes = sum(lens[i] for i in range(C)) * tok_bytes

    def timed(fn, steps, warm):
        for _ in range(warm):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    def attn(b):
        if a.fp8:
            return lambda: pa.attention_fp8(b["out"], b["q"], dw.k_cache, dw.v_cache, b["block_table"],
                                            b["seq_lens"], b["query_start_loc"], max_query_len=b["max_query_len"],
                                            max_seq_len=b["max_seq_len"], scale=sp.scale, k_scale=wl.k_scale,
                                            v_scale=wl.v_scale, workspace=st.workspace, stream=stream)
        return lambda: pa.attention(b["out"], b["q"], dw.k_cache, dw.v_cache, b["block_table"], b["seq_lens"],
                                    b["query_start_loc"], max_query_len=b["max_query_len"],
                                    max_seq_len=b["max_seq_len"], scale=sp.scale, workspace=st.workspace,
                                    stream=stream)

    whole = dict(q=st.q, out=st.out, block_table=st.block_table, seq_lens=st.seq_lens,
                 query_start_loc=st.query_start_loc, max_query_len=st.max_query_len, max_seq_len=st.max_seq_len)
    pre = _sub_batch(st, None, list(range(C)), dev)
    dec = _sub_batch(st, None, list(range(C, len(lens))), dev)
    steps = max(10, a.steps // 10)
    pa.read_device_errors(clear=True)
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    step_ms = timed(lambda: dw.run_step(st, stream=stream), steps, a.warmup)
    attn_ms = timed(attn(whole), steps, a.warmup)
    pre_ms = timed(attn(pre), steps, a.warmup)
    dec_ms = timed(attn(dec), steps, a.warmup)
    clk = clocks.stop()
    if pa.read_device_errors(clear=True):
        raise RuntimeError("device error flags set")
    hbm, tflops_peak, src = _peaks()
    pre_tf = pf_flops / (pre_ms * 1e-3) / 1e12
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    t_star = max(pf_flops / (tflops_peak * 1e12), (dec_bytes + pf_kv_bytes) / (hbm * 1e9)) * 1e3
    line = {
        "metric": "mixed chunked-prefill + decode attention (8 x 512-query chunks + 248 decodes)"
                  + (" over an E4M3 cache" if a.fp8 else ""),
        "value": t_star / attn_ms, "unit": "fraction of max(flops / tensor peak, bytes / HBM peak) roofline time",
        "n_gpus": 1, "steps": steps, "warmup": a.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "dtype": "e4m3 cache, f16 MMA operands" if a.fp8 else "bf16", "data": "synthetic",
        "config": {"workload": "mixed_prefill_decode_bf16: 8 chunks x 512 queries, prior context U[0, 4096]; "
                               "248 decodes, L ~ U[256, 4096]; 32 q / 8 kv heads, head_dim 128, block 16"
                               + ("; E4M3 K/V cache (scales 2^-6)" if a.fp8 else ""),
                   "prefill_gflop": pf_flops / 1e9, "decode_kv_bytes": dec_bytes, "seed": wl.seed},
        "attention_ms": attn_ms, "roofline_time_ms": t_star,
        "execution": "one pa_attention call: the decode kernels on 3/5 of the SMs on a side stream beside the "
                     "prefill kernel, whose CTAs also take the rest of the GPU once the decode CTAs are done; "
                     "the two parts below are the same call on each sub-batch alone",
        "prefill": {"ms": pre_ms, "tflops": pre_tf, "peak_tflops": tflops_peak, "frac": pre_tf / tflops_peak,
                    "bound": "tensor", "kernel": "prefill_tc_kernel (tcgen05" +
                    (", E4M3 codes converted to f16 tiles by the producer warps)" if a.fp8 else ")")},
        "decode": {"ms": dec_ms, "gbs": dec_gbs, "peak_gbs": hbm, "frac": dec_gbs / hbm, "bound": "hbm"},
        "peak_source": src, "clocks": clk,
    }
    return line


def run_mixed(a):
    print(json.dumps(mixed_line(a)))
    return 0


def run_prefill(a):
    """The mixed batch's 8 chunked-prefill requests alone, as one prefill launch over all SMs
    (pa_attention_fixed_scratch keeps every kernel on the caller's stream) and through
    pa_attention (two prefill launches sharing one pair counter, the first on the SMs a
    decode kernel would leave): the tensor-core kernel's own roofline fraction."""
    import torch

    import paged_kv_cache_161_gb300 as pa
    import workloads
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    wl = workloads.build(5)
    if a.fp8:
        wl = workloads.with_fp8_cache(wl)
    sp = wl.spec
    dw = DeviceWorkload(wl, device=dev)
    dw.run_setup()
    st = dw.prepare_step()
    dw.run_step(st)  # writes the chunks' own K/V
    stream = torch.cuda.current_stream(dev)
    C = wl.meta["chunks"]
    b = _sub_batch(st, None, list(range(C)), dev)
    lens = b["seq_lens"].cpu().tolist()
    qlens = torch.diff(b["query_start_loc"].cpu()).tolist()
    flops = sum(4.0 * sp.head_dim * sp.num_heads * sum(lens[i] - qlens[i] + j + 1 for j in range(qlens[i]))
                for i in range(C))
    kw = dict(max_query_len=b["max_query_len"], max_seq_len=b["max_seq_len"], scale=sp.scale, stream=stream)
    if a.fp8:
        one = lambda: pa.attention_fp8(b["out"], b["q"], dw.k_cache, dw.v_cache, b["block_table"], b["seq_lens"],  # noqa: E731
                                       b["query_start_loc"], k_scale=wl.k_scale, v_scale=wl.v_scale,
                                       workspace=st.workspace, **kw)
        single = None
    else:
        one = lambda: pa.attention(b["out"], b["q"], dw.k_cache, dw.v_cache, b["block_table"], b["seq_lens"],  # noqa: E731
                                   b["query_start_loc"], workspace=st.workspace, **kw)
        single = lambda: pa.attention_fixed_scratch(b["out"], b["q"], dw.k_cache, dw.v_cache, b["block_table"],  # noqa: E731
                                                    b["seq_lens"], b["query_start_loc"], **kw)

    def timed(fn, steps, warm):
        for _ in range(warm):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    steps = max(10, a.steps // 10)
    pa.read_device_errors(clear=True)
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    ms = timed(single if single is not None else one, steps, a.warmup)
    ms_two = timed(one, steps, a.warmup) if single is not None else None
    clk = clocks.stop()
    if pa.read_device_errors(clear=True):
        raise RuntimeError("device error flags set")
    hbm, tflops_peak, src = _peaks()
    tf = flops / (ms * 1e-3) / 1e12
    line = {
        "metric": "chunked-prefill attention (8 x 512-query chunks of the mixed batch), TFLOP/s"
                  + (" over an E4M3 cache" if a.fp8 else ""),
        "value": tf, "unit": "TFLOP/s", "n_gpus": 1, "steps": steps, "warmup": a.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "e4m3 cache, f16 MMA operands" if a.fp8 else "bf16", "data": "synthetic",
        "config": {"workload": "the mixed batch's prefill part: 8 chunks x 512 queries, prior context U[0, 4096], "
                               "32 q / 8 kv heads, head_dim 128, block 16", "gflop": flops / 1e9, "seed": wl.seed},
        "roofline": {"bound": "tensor", "achieved": tf, "peak": tflops_peak, "unit": "TFLOP/s",
                     "frac": tf / tflops_peak, "peak_source": src,
                     "kernel": "prefill_tc_kernel, one launch of one CTA per SM" if single is not None else
                               "prefill_tc_kernel (pa_attention_fp8)"},
        "clocks": clk,
    }
    if ms_two is not None:
        line["through_pa_attention"] = {"ms": ms_two, "tflops": flops / (ms_two * 1e-3) / 1e12,
                                        "frac": flops / (ms_two * 1e-3) / 1e12 / tflops_peak,
                                        "launches": "two prefill launches sharing one pair counter"}
    print(json.dumps(line))
    return 0


def secondary_line(a):
    """MHA decode (attention only) or shared-prefix sampling (copy-on-write copies, write,
    attention): per-operation times and bytes on one GPU, device-resident inputs."""
    import torch

    import paged_kv_cache_161_gb300 as pa
    import workloads
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    cfg = 2 if a.workload == "mha_decode" else 4
    wl = workloads.build(cfg)
    sp = wl.spec
    dw = DeviceWorkload(wl, device=dev)
    dw.run_setup()
    st = dw.prepare_step()
    stream = torch.cuda.current_stream(dev)
    hbm, _, src = _peaks()

    def timed(fn, steps, warm):
        for _ in range(warm):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    steps = max(20, a.steps // 4)
    pa.read_device_errors(clear=True)
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    attn = lambda: pa.attention(st.out, st.q, dw.k_cache, dw.v_cache, st.block_table, st.seq_lens,  # noqa: E731
                                st.query_start_loc, max_query_len=st.max_query_len, max_seq_len=st.max_seq_len,
                                scale=sp.scale, workspace=st.workspace, stream=stream)
    attn_ms = timed(attn, steps, a.warmup)
    lens = st.seq_lens.cpu().long()
    logical = int(lens.sum()) * sp.kv_token_bytes
    line = {"metric": f"{wl.name}: attention K/V GB/s", "n_gpus": 1, "steps": steps, "warmup": a.warmup,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic", "peak_gbs": hbm, "peak_source": src,
            "attention_ms": attn_ms, "attention_gbs_logical": logical / (attn_ms * 1e-3) / 1e9,
            "config": {"workload": wl.name, "requests": int(lens.numel()), "kv_bytes_logical": logical,
                       "seed": wl.seed}}
    if cfg == 4:
        # unique bytes: each physical block read once however many samples share it
        table = st.block_table.cpu()
        B = sp.block_size
        seen = set()
        uniq_tokens = 0
        for i in range(table.shape[0]):
            L = int(lens[i])
            for j in range((L + B - 1) // B):
                b = int(table[i, j])
                if b not in seen:
                    seen.add(b)
                    uniq_tokens += B if (j + 1) * B <= L else L - j * B
        uniq = uniq_tokens * sp.kv_token_bytes
        pairs = torch.cat([torch.from_numpy(c.reshape(-1, 2)) for c in dw.phase_copies if len(c)]).to(dev)
        cp_ms = timed(lambda: pa.copy_blocks(dw.k_cache, dw.v_cache, pairs, stream=stream), steps, a.warmup)
        block_bytes = B * sp.num_kv_heads * sp.head_dim * 2 * 2  # K and V
        cp_bytes = 2 * int(pairs.shape[0]) * block_bytes  # read + write
        wr_ms = timed(lambda: pa.kv_write(st.k_new, st.v_new, dw.k_cache, dw.v_cache, st.slot_mapping,
                                          stream=stream), steps, a.warmup)
        wr_bytes = 2 * int(st.slot_mapping.shape[0]) * sp.kv_token_bytes
        # grouped decode: each group's shared prefix read once, members' own tails separately
        seqs = [s for s, _ in wl.step.batch]
        sg, gr, sl = dw.bm.batch_groups(seqs, 4)
        sg_d, gr_d, sl_d = (torch.from_numpy(x).to(dev) for x in (sg, gr, sl))
        gws = torch.zeros(pa.attention_grouped_workspace_size(len(seqs), len(sl), sp.num_heads, sp.num_kv_heads,
                                                              sp.head_dim), dtype=torch.uint8, device=dev)
        gout = torch.empty_like(st.out)
        grp = lambda: pa.attention_grouped(gout, st.q, dw.k_cache, dw.v_cache, st.block_table, st.seq_lens,  # noqa: E731
                                           st.query_start_loc, sg_d, gr_d, sl_d, max_seq_len=st.max_seq_len,
                                           scale=sp.scale, workspace=gws, stream=stream)
        grp_ms = timed(grp, steps, a.warmup)
        shared_tok = sum(int(sl[g]) for g in range(len(sl)))
        own_tok = sum(int(lens[i]) - (int(sl[sg[i]]) if sg[i] >= 0 else 0) for i in range(len(seqs)))
        grp_read = (shared_tok + own_tok) * sp.kv_token_bytes
        line.update({
            "grouped": {"groups": int(len(sl)), "members": int((sg >= 0).sum()), "ms": grp_ms,
                        "speedup_vs_attention": attn_ms / grp_ms,
                        "kv_bytes_read": grp_read, "gbs_read": grp_read / (grp_ms * 1e-3) / 1e9,
                        "frac_read": grp_read / (grp_ms * 1e-3) / 1e9 / hbm,
                        "gbs_unique": uniq / (grp_ms * 1e-3) / 1e9, "frac_unique": uniq / (grp_ms * 1e-3) / 1e9 / hbm},
            "attention_gbs_unique": uniq / (attn_ms * 1e-3) / 1e9, "frac_unique": uniq / (attn_ms * 1e-3) / 1e9 / hbm,
            "copy_blocks": {"pairs": int(pairs.shape[0]), "ms": cp_ms, "gbs": cp_bytes / (cp_ms * 1e-3) / 1e9,
                            "bytes": cp_bytes},
            "kv_write": {"tokens": int(st.slot_mapping.shape[0]), "ms": wr_ms,
                         "gbs": wr_bytes / (wr_ms * 1e-3) / 1e9},
        })
        line["config"]["kv_bytes_unique"] = uniq
    else:
        line["frac_logical"] = line["attention_gbs_logical"] / hbm
    line["clocks"] = clocks.stop()
    if pa.read_device_errors(clear=True):
        raise RuntimeError("device error flags set")
    return line


def run_secondary(a):
    print(json.dumps(secondary_line(a)))
    return 0


def _host_admission_ms(wl, reps=5):
    """Host block accounting of the step alone (C++ manager): the admissions (lookups with
    prefix caching) and token appends of every request, median of ``reps`` fresh runs."""
    import paged_kv_cache_161_gb300 as pa

    times = []
    for _ in range(reps):
        bm = pa.BlockManager(wl.num_blocks, wl.spec.block_size, wl.free_order)
        if wl.prefix_caching:
            bm.enable_prefix_caching()

        def run(ops):
            for op in ops:
                if op[0] == "prompt":
                    s, n = op[1], op[2]
                    toks = wl.tokens(s, 0, n)
                    if wl.prefix_caching:
                        hit = bm.add_seq_cached(s, toks, n - 1)
                        bm.append_tokens(s, toks[hit:])
                    else:
                        bm.add_seq(s)
                        bm.append(s, n)
                elif op[0] == "free":
                    bm.free_seq(op[1])

        for ph in wl.setup:
            run(ph.ops)
        t0 = time.perf_counter()
        run(wl.step.ops)
        times.append((time.perf_counter() - t0) * 1e3)
    return sorted(times)[len(times) // 2]


def run_system_prompt(a):
    """Many requests sharing one system prompt, admitted as one chunked-prefill batch, with
    and without prefix caching: each step is one pa_write_attention call (the write of the
    computed tokens, then prefill attention over the whole prompt through the block table)."""
    import torch

    import paged_kv_cache_161_gb300 as pa
    import workloads
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    hbm, tflops_peak, src = _peaks()

    def timed(fn, steps, warm):
        for _ in range(warm):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    steps = max(10, a.steps // 20)
    res = {}
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    for caching in (True, False):
        wl = workloads.system_prompt("full", caching=caching)
        sp = wl.spec
        dw = DeviceWorkload(wl, device=dev)
        dw.run_setup()
        st = dw.prepare_step()
        pa.read_device_errors(clear=True)
        ms = timed(lambda: dw.run_step(st, stream=stream, fused=True), steps, a.warmup)
        if pa.read_device_errors(clear=True):
            raise RuntimeError("device error flags set")
        lens = st.seq_lens.cpu().tolist()
        qlens = torch.diff(st.query_start_loc.cpu()).tolist()
        pairs = sum(q * (L - q) + q * (q + 1) // 2 for L, q in zip(lens, qlens))
        flops = 4.0 * sp.head_dim * sp.num_heads * pairs
        tf = flops / (ms * 1e-3) / 1e12
        res[caching] = {"ms": ms, "computed_tokens": int(sum(qlens)), "prompt_tokens": int(sum(lens)),
                        "gflop": flops / 1e9, "tflops": tf, "frac_of_bf16_peak": tf / tflops_peak,
                        "host_admission_ms": _host_admission_ms(wl),
                        "kv_write_bytes": 2 * int(sum(qlens)) * sp.kv_token_bytes}
        if caching:
            res[caching]["prefix_stats"] = dict(zip(("cached_blocks", "hit_blocks", "evictions"),
                                                    dw.bm.prefix_stats()))
        meta = wl.meta
        del dw, st
        torch.cuda.empty_cache()
    clk = clocks.stop()
    c, u = res[True], res[False]
    line = {
        "metric": "system-prompt batch: prompt tokens/s with prefix caching (64 requests, 2040-token shared prompt)",
        "value": c["prompt_tokens"] / (c["ms"] * 1e-3), "unit": "prompt tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": a.warmup, "ms_per_step": c["ms"], "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "system_prompt_bf16: 64 requests = one 2040-token system prompt (computed once by a "
                               "warm request that then ended) + user text U[64, 512]; 32 q / 8 kv heads, head_dim "
                               "128, block 16", "requests": meta["requests"], "system_len": meta["system_len"],
                   "seed": wl.seed},
        "cached": c, "uncached": u, "speedup": u["ms"] / c["ms"],
        "uncached_prompt_tokens_per_s": u["prompt_tokens"] / (u["ms"] * 1e-3),
        "roofline": {"bound": "tensor", "achieved": c["tflops"], "peak": tflops_peak, "unit": "TFLOP/s",
                     "frac": c["frac_of_bf16_peak"], "peak_source": src,
                     "kernel": "pa_write_attention: kv_write + prefill_tc_kernel (tcgen05)"},
        "clocks": clk,
    }
    print(json.dumps(line))
    return 0


def run_fp8_decode(a):
    """The GQA batch-256 decode step over an FP8 (E4M3) cache: pa_kv_write_fp8 of the 256 new
    tokens, then pa_attention_fp8 (split-K + merge over 1-byte K/V). Reports the K/V bytes
    the attention reads per second (half of bf16's for the same tokens) and tokens/s; the
    bf16 step of the same batch is timed in the same run for comparison."""
    import torch

    import paged_kv_cache_161_gb300 as pa
    import workloads
    from paged_kv_cache_161_gb300.device_workload import DeviceWorkload

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    hbm, _, src = _peaks()

    def timed(fn, steps, warm):
        for _ in range(warm):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    steps = max(50, a.steps // 2)
    res = {}
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    for name, wl in (("fp8", workloads.with_fp8_cache(workloads.build(CONFIG_ID))), ("bf16", workloads.build(CONFIG_ID))):
        sp = wl.spec
        dw = DeviceWorkload(wl, device=dev, table_width=E2E_TABLE_WIDTH)
        dw.run_setup()
        st = dw.prepare_step()
        pa.read_device_errors(clear=True)
        step_ms = timed(lambda: dw.run_step(st, stream=stream), steps, a.warmup)
        attn_ms = timed(lambda: dw._attend(st, stream=stream), steps, a.warmup)
        if pa.read_device_errors(clear=True):
            raise RuntimeError("device error flags set")
        tokens = int(st.seq_lens.sum().item())
        el = 1 if name == "fp8" else 2
        kv_bytes = tokens * 2 * sp.num_kv_heads * sp.head_dim * el
        res[name] = {"step_ms": step_ms, "attention_ms": attn_ms, "kv_bytes": kv_bytes,
                     "attention_gbs": kv_bytes / (attn_ms * 1e-3) / 1e9,
                     "frac_of_hbm": kv_bytes / (attn_ms * 1e-3) / 1e9 / hbm,
                     "tokens_per_s": int(st.seq_lens.shape[0]) / (step_ms * 1e-3)}
        meta_seed = wl.seed
        del dw, st
        torch.cuda.empty_cache()
    clk = clocks.stop()
    f, b = res["fp8"], res["bf16"]
    line = {
        "metric": "paged decode attention over an FP8 (E4M3) KV cache: K/V GB/s and tokens/s, batch 256",
        "value": f["kv_bytes"] / (f["step_ms"] * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": 1, "steps": steps,
        "warmup": a.warmup, "ms_per_step": f["step_ms"], "higher_is_better": True, "dtype": "fp8_e4m3 cache, bf16 q/out",
        "data": "synthetic",
        "config": {"workload": "gqa_bf16_decode_b256 over an E4M3 cache (k_scale = v_scale = 2^-6): 256 requests, "
                               "32 q / 8 kv heads, head_dim 128, block 16, lognormal context", "seed": meta_seed},
        "fp8": f, "bf16": b, "speedup_step": b["step_ms"] / f["step_ms"],
        "speedup_attention": b["attention_ms"] / f["attention_ms"],
        "roofline": {"bound": "hbm", "achieved": f["attention_gbs"], "peak": hbm, "unit": "GB/s",
                     "frac": f["frac_of_hbm"], "peak_source": src,
                     "kernel": "pa_attention_fp8 decode (split-K + merge, 1-byte K/V)"},
        "clocks": clk,
    }
    print(json.dumps(line))
    return 0


def run_swap(a):
    """Swap bandwidth: 8192 scattered blocks (16 tokens x 8 KV heads x 128 dims bf16, K and V:
    512 MiB) moved GPU -> pinned CPU pool and back by pa_swap_blocks (one launch each way),
    against a contiguous copy of the same bytes over the same link (cudaMemcpyAsync through
    torch) timed in the same run."""
    import torch

    import paged_kv_cache_161_gb300 as pa

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    NB, NC, B, H, D, N = 40000, 16384, 16, 8, 128, 8192
    g = torch.Generator().manual_seed(161008)
    gk = torch.empty((NB, B, H, D), dtype=torch.bfloat16, device=dev).normal_()
    gv = torch.empty_like(gk).normal_()
    ck = torch.empty((NC, B, H, D), dtype=torch.bfloat16).pin_memory()
    cv = torch.empty_like(ck).pin_memory()
    src = torch.randperm(NB, generator=g)[:N]
    dst = torch.randperm(NC, generator=g)[:N]
    out_map = torch.stack([src, dst], 1).to(dev)
    in_map = torch.stack([dst, torch.randperm(NB, generator=g)[:N]], 1).to(dev)
    nbytes = 2 * N * B * H * D * 2

    def timed(fn, steps, warm):
        for _ in range(warm):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    steps = max(5, a.steps // 60)
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    pa.read_device_errors(clear=True)
    out_ms = timed(lambda: pa.swap_blocks(gk, gv, ck, cv, out_map, stream=stream), steps, a.warmup)
    in_ms = timed(lambda: pa.swap_blocks(ck, cv, gk, gv, in_map, stream=stream), steps, a.warmup)
    if pa.read_device_errors(clear=True):
        raise RuntimeError("device error flags set")
    flat_d = gk.view(-1)[: nbytes // 2]
    flat_h = torch.empty(nbytes // 2, dtype=torch.bfloat16).pin_memory()
    d2h_ms = timed(lambda: flat_h.copy_(flat_d, non_blocking=True), steps, a.warmup)
    h2d_ms = timed(lambda: flat_d.copy_(flat_h, non_blocking=True), steps, a.warmup)
    clk = clocks.stop()
    gbs = lambda ms: nbytes / (ms * 1e-3) / 1e9  # noqa: E731
    line = {
        "metric": "swap_blocks: scattered KV blocks between the GPU pool and a pinned CPU pool, GB/s",
        "value": gbs(out_ms), "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": a.warmup,
        "ms_per_step": out_ms, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{N} random blocks of 16 x 8 x 128 bf16 (K and V, {nbytes / 2**20:.0f} MiB) from a "
                               f"{NB}-block GPU pool to a {NC}-block pinned pool and back"},
        "swap_out": {"ms": out_ms, "gbs": gbs(out_ms), "frac_of_contiguous_copy": d2h_ms / out_ms},
        "swap_in": {"ms": in_ms, "gbs": gbs(in_ms), "frac_of_contiguous_copy": h2d_ms / in_ms},
        "contiguous_copy": {"d2h_ms": d2h_ms, "d2h_gbs": gbs(d2h_ms), "h2d_ms": h2d_ms, "h2d_gbs": gbs(h2d_ms)},
        "roofline": {"bound": "link", "achieved": gbs(out_ms), "peak": gbs(d2h_ms), "unit": "GB/s",
                     "frac": d2h_ms / out_ms,
                     "peak_source": "a contiguous device-to-host copy of the same bytes, same run"},
        "clocks": clk,
    }
    print(json.dumps(line))
    return 0


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    a = _args(argv)
    if a.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # started without a launcher: run this command again as a.gpus ranks, one per GPU
        if a.workload != "gqa_decode":
            raise SystemExit("--gpus > 1 runs the default workload (gqa_decode) only")
        return subprocess.call(launch_command(a.gpus, argv))
    if a.impl == "reference":
        return run_reference(a)
    if a.workload == "mixed":
        return run_mixed(a)
    if a.workload == "prefill":
        return run_prefill(a)
    if a.workload in ("mha_decode", "shared_prefix"):
        return run_secondary(a)
    if a.workload == "system_prompt":
        return run_system_prompt(a)
    if a.workload == "gqa_decode_fp8":
        return run_fp8_decode(a)
    if a.workload == "swap":
        return run_swap(a)
    return run_ours(a)


if __name__ == "__main__":
    sys.exit(main())
