"""Execute a seeded workload on the GPU through the C ABI.

The block manager is the library's C++ one (pa_bm_*), the copies, writes and attention
are its kernels; this module only moves the generator's values to the device and hands
the library's outputs from one call to the next. A phase runs as the workload script
defines: block-manager operations, then pa_copy_blocks of the emitted pairs, then
pa_kv_write of the appended tokens, then (for the step) pa_attention over the batch --
or, for a step whose appended tokens are exactly its query tokens, pa_write_attention.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import (BlockManager, attention, attention_fp8, attention_workspace_size, copy_blocks, kv_write,
               kv_write_fp8, swap_blocks, write_attention)


def storage_to_torch(a: np.ndarray) -> torch.Tensor:
    """float32 arrays stay float32; uint16 arrays hold bfloat16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


def torch_to_storage(t: torch.Tensor) -> np.ndarray:
    """float32 -> float32; bfloat16 -> uint16 bit patterns; float8_e4m3fn -> uint8 codes."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


@dataclass
class StepInputs:
    """Device tensors of one timed step (write + copies + attention)."""
    slot_mapping: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    block_mapping: torch.Tensor
    q: torch.Tensor
    out: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    query_start_loc: torch.Tensor
    max_query_len: int
    max_seq_len: int
    workspace: torch.Tensor


class DeviceWorkload:
    def __init__(self, wl, device="cuda", table_width: int | None = None):
        self.wl = wl
        sp = wl.spec
        self.device = torch.device(device)
        self.bm = BlockManager(wl.num_blocks, sp.block_size, wl.free_order)
        if wl.prefix_caching:
            self.bm.enable_prefix_caching()
        if wl.cpu_blocks:
            self.bm.enable_swap(wl.cpu_blocks, wl.cpu_free_order)
        self.dtype = torch.float32 if sp.dtype == "f32" else torch.bfloat16
        shape = (wl.num_blocks, sp.block_size, sp.num_kv_heads, sp.head_dim)
        self.fp8 = wl.kv_cache == "fp8_e4m3"
        cache_dtype = torch.float8_e4m3fn if self.fp8 else self.dtype
        self.k_cache = torch.zeros(shape, dtype=cache_dtype, device=self.device)
        self.v_cache = torch.zeros(shape, dtype=cache_dtype, device=self.device)
        if wl.cpu_blocks:  # the CPU pool: pinned host memory, read and written by the swap kernel
            cshape = (wl.cpu_blocks,) + shape[1:]
            self.k_cpu = torch.zeros(cshape, dtype=cache_dtype).pin_memory()
            self.v_cpu = torch.zeros(cshape, dtype=cache_dtype).pin_memory()
        self.phase_swaps: list = []
        self.table_width = table_width
        self.phase_slots: list = []
        self.phase_copies: list = []

    # -- block manager side ------------------------------------------------------
    def _append(self, s, n):
        if self.wl.prefix_caching:
            return self.bm.append_tokens(s, self.wl.tokens(s, self.bm.seq_len(s), n))
        return self.bm.append(s, n)

    def _ops(self, phase):
        """Run a phase's operations on the C++ block manager: (slots, copy pairs, appended
        ranges (seq, start, n) in operation order)."""
        slots, apps, swaps = [], [], []
        for op in phase.ops:
            if op[0] == "add":
                self.bm.add_seq(op[1])
            elif op[0] == "fork":
                self.bm.fork(op[1], op[2])
            elif op[0] == "append":
                apps.append((op[1], self.bm.seq_len(op[1]), op[2]))
                slots.append(self._append(op[1], op[2]))
            elif op[0] == "prompt":
                s, n = op[1], op[2]
                if self.wl.prefix_caching:
                    hit = self.bm.add_seq_cached(s, self.wl.tokens(s, 0, n), n - 1)
                else:
                    self.bm.add_seq(s)
                    hit = 0
                apps.append((s, hit, n - hit))
                slots.append(self._append(s, n - hit))
            elif op[0] == "fill":
                n = self.bm.num_free() * self.wl.spec.block_size
                apps.append((op[1], 0, n))
                slots.append(self._append(op[1], n))
            elif op[0] == "free":
                self.bm.free_seq(op[1])
            elif op[0] == "swap_out":
                swaps.append(("out", self.bm.swap_out(list(op[1]))))
            elif op[0] == "swap_in":
                swaps.append(("in", self.bm.swap_in(list(op[1]))))
        slots = np.concatenate(slots) if slots else np.zeros(0, np.int64)
        copies = self.bm.take_copies()
        self.phase_slots.append(slots)
        self.phase_copies.append(copies)
        self.phase_swaps.append(swaps)
        self._pending_swaps = swaps
        return slots, copies, apps

    def _apply_swaps(self, swaps, stream=None):
        for direction, pairs in swaps:
            if not len(pairs):
                continue
            m = torch.from_numpy(np.ascontiguousarray(pairs)).to(self.device)
            if direction == "out":
                swap_blocks(self.k_cache, self.v_cache, self.k_cpu, self.v_cpu, m, stream=stream)
            else:
                swap_blocks(self.k_cpu, self.v_cpu, self.k_cache, self.v_cache, m, stream=stream)

    def _values(self, apps):
        if not apps:
            sp = self.wl.spec
            z = torch.zeros((0, sp.num_kv_heads, sp.head_dim), dtype=self.dtype)
            return z, z
        vals = self.wl.kv_many(apps)
        k = np.concatenate([kv[0] for kv in vals])
        v = np.concatenate([kv[1] for kv in vals])
        return storage_to_torch(k), storage_to_torch(v)

    # -- phases --------------------------------------------------------------------
    def run_setup(self):
        """All untimed phases: operations, copies, writes."""
        for ph in self.wl.setup:
            slots, copies, apps = self._ops(ph)
            k, v = self._values(apps)
            if len(copies):
                copy_blocks(self.k_cache, self.v_cache, torch.from_numpy(copies).to(self.device))
            self._apply_swaps(self._pending_swaps)
            if len(slots):
                self._write(k.to(self.device), v.to(self.device), torch.from_numpy(slots).to(self.device))

    def prepare_step(self) -> StepInputs:
        """Run the step's block-manager operations and stage its inputs on the device."""
        wl = self.wl
        sp = wl.spec
        slots, copies, apps = self._ops(wl.step)
        self._apply_swaps(self._pending_swaps)  # (a step script normally has none)
        self.step_appends = apps
        k, v = self._values(apps)
        batch = wl.step.batch or []
        seqs = [s for s, _ in batch]
        nblk = [int(np.ceil(self.bm.seq_len(s) / sp.block_size)) for s in seqs]
        width = self.table_width or max(nblk + [1])
        table, lens = self.bm.batch_tables(seqs, width)
        appended = {}
        for s, _, n in apps:
            appended[s] = appended.get(s, 0) + n
        qranges = wl.step_queries({s: self.bm.seq_len(s) for s in seqs}, appended)
        q = np.concatenate([wl.q(s, a, n) for s, a, n in qranges]) if qranges else \
            np.zeros((0, sp.num_heads, sp.head_dim), np.float32 if sp.dtype == "f32" else np.uint16)
        qsl = np.zeros(len(batch) + 1, np.int32)
        qsl[1:] = np.cumsum([n for _, _, n in qranges])
        dev = self.device
        qt = storage_to_torch(q).to(dev)
        ws = torch.empty(attention_workspace_size(len(batch), sp.num_heads, sp.num_kv_heads, sp.head_dim),
                         dtype=torch.uint8, device=dev)
        return StepInputs(
            slot_mapping=torch.from_numpy(slots).to(dev),
            k_new=k.to(dev), v_new=v.to(dev),
            block_mapping=torch.from_numpy(copies.reshape(-1, 2)).to(dev),
            q=qt, out=torch.empty_like(qt),
            block_table=torch.from_numpy(table).to(dev),
            seq_lens=torch.from_numpy(lens).to(dev),
            query_start_loc=torch.from_numpy(qsl).to(dev),
            max_query_len=int(max([n for _, _, n in qranges] + [0])),
            max_seq_len=int(lens.max()) if len(lens) else 0,
            workspace=ws,
        )

    def _write(self, k, v, slots, stream=None):
        if self.fp8:
            kv_write_fp8(k, v, self.k_cache, self.v_cache, slots, self.wl.k_scale, self.wl.v_scale, stream=stream)
        else:
            kv_write(k, v, self.k_cache, self.v_cache, slots, stream=stream)

    def _attend(self, st: StepInputs, stream=None):
        kw = dict(max_query_len=st.max_query_len, max_seq_len=st.max_seq_len, scale=self.wl.spec.scale,
                  workspace=st.workspace, stream=stream)
        if self.fp8:
            attention_fp8(st.out, st.q, self.k_cache, self.v_cache, st.block_table, st.seq_lens, st.query_start_loc,
                          k_scale=self.wl.k_scale, v_scale=self.wl.v_scale, **kw)
        else:
            attention(st.out, st.q, self.k_cache, self.v_cache, st.block_table, st.seq_lens, st.query_start_loc,
                      **kw)

    def fusable(self, st: StepInputs) -> bool:
        """The step appends exactly its query tokens (row t of k_new belongs to query row t)."""
        return st.q.shape[0] > 0 and st.slot_mapping.shape[0] == st.q.shape[0]

    def run_step(self, st: StepInputs, stream=None, fused: bool = False):
        """The hot path of one step: copies, write, attention (all on the device).

        ``fused``: the write and the attention as one pa_write_attention call (the step
        must be fusable; an FP8 cache has no fused call and runs the two)."""
        sp = self.wl.spec
        if st.block_mapping.shape[0]:
            copy_blocks(self.k_cache, self.v_cache, st.block_mapping, stream=stream)
        if fused and not self.fp8:
            if not self.fusable(st):
                raise ValueError("this step's appended tokens are not its query tokens")
            write_attention(st.out, st.q, st.k_new, st.v_new, st.slot_mapping, self.k_cache, self.v_cache,
                            st.block_table, st.seq_lens, st.query_start_loc, max_query_len=st.max_query_len,
                            max_seq_len=st.max_seq_len, scale=sp.scale, workspace=st.workspace, stream=stream)
            return st.out
        if st.slot_mapping.shape[0]:
            self._write(st.k_new, st.v_new, st.slot_mapping, stream=stream)
        if st.q.shape[0]:
            self._attend(st, stream=stream)
        return st.out
