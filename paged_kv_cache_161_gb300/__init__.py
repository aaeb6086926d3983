"""GB300 (sm_103a) paged-KV-cache hot path: a thin ctypes binding over libpa_gb300.so.

Names follow the C ABI in include/pa.h (pa_kv_write -> kv_write, ...). The binding only
checks tensors and marshals pointers, sizes and the current CUDA stream; every step of
the path runs in the library's kernels. PyTorch provides device memory and streams.

The library is built in-tree by ``python paged_kv_cache_161_gb300/build.py`` (or the
repository's ``__graft_entry__.build()``). Importing this package without it raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libpa_gb300.so")

__all__ = [
    "PAError",
    "BlockManager",
    "kv_write",
    "copy_blocks",
    "swap_blocks",
    "attention",
    "write_attention",
    "attention_grouped",
    "attention_grouped_workspace_size",
    "kv_write_fp8",
    "attention_fp8",
    "attention_workspace_size",
    "read_device_errors",
    "lib",
    "LIB_PATH",
]

PA_F32, PA_BF16, PA_FP8_E4M3 = 0, 1, 2
PA_DEVERR = {"slot_range": 0x1, "block_range": 0x2, "seq_range": 0x4, "timeout": 0x8, "slot_mismatch": 0x10}

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python paged_kv_cache_161_gb300/build.py` "
        "(there is no fallback path)")

lib = ctypes.CDLL(LIB_PATH)

_p, _i, _i64, _sz, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_sig = {
    "pa_status_string": (ctypes.c_char_p, [_i]),
    "pa_last_cuda_error": (_i, []),
    "pa_read_device_errors": (_i, [ctypes.POINTER(ctypes.c_uint), _i]),
    "pa_kv_write": (_i, [_p, _p, _p, _p, _p, _i64, _i64, _i, _i, _i, _i, _p]),
    "pa_copy_blocks": (_i, [_p, _p, _p, _i64, _i64, _i, _i, _i, _i, _p]),
    "pa_attention_workspace_size": (_i, [_i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "pa_attention": (_i, [_p, _p, _p, _p, _p, _i, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i64, _f, _i, _p,
                          _sz, _p]),
    "pa_write_attention": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _i, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i,
                                _i64, _f, _i, _p, _sz, _p]),
    "pa_kv_write_fp8": (_i, [_p, _p, _i, _p, _p, _p, _i64, _i64, _i, _i, _i, _f, _f, _p]),
    "pa_attention_fp8": (_i, [_p, _p, _p, _p, _p, _i, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i64, _f, _f, _f,
                              _p, _sz, _p]),
    "pa_swap_blocks": (_i, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i, _i, _i, _i, _p]),
    "pa_attention_fixed_scratch": (_i, [_p, _p, _p, _p, _p, _i, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i64, _f,
                                        _i, _p]),
    "pa_attention_grouped_workspace_size": (_i, [_i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "pa_attention_grouped": (_i, [_p, _p, _p, _p, _p, _i, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i64, _f, _i, _p, _p,
                                  _p, _i, _p, _sz, _p]),
    "pa_bm_batch_groups": (_i, [_p, _p, _i64, _i, _p, _p, _p, _i64, ctypes.POINTER(_i64)]),
    "pa_bm_enable_swap": (_i, [_p, _i64, _p]),
    "pa_bm_swap_out": (_i, [_p, _p, _i64, _p, _i64, ctypes.POINTER(_i64)]),
    "pa_bm_swap_in": (_i, [_p, _p, _i64, _p, _i64, ctypes.POINTER(_i64)]),
    "pa_bm_is_swapped": (_i, [_p, _i64]),
    "pa_bm_num_free_cpu": (_i64, [_p]),
    "pa_bm_cpu_ref_count": (_i, [_p, _i64]),
    "pa_bm_create": (_p, [_i64, _i, _p]),
    "pa_bm_destroy": (None, [_p]),
    "pa_bm_add_seq": (_i, [_p, _i64]),
    "pa_bm_append": (_i, [_p, _i64, _i64, _p]),
    "pa_bm_append_batch": (_i, [_p, _p, _p, _i64, _p, _p]),
    "pa_bm_fork": (_i, [_p, _i64, _i64]),
    "pa_bm_free_seq": (_i, [_p, _i64]),
    "pa_bm_seq_len": (_i64, [_p, _i64]),
    "pa_bm_num_seq_blocks": (_i64, [_p, _i64]),
    "pa_bm_ref_count": (_i, [_p, _i64]),
    "pa_bm_num_free": (_i64, [_p]),
    "pa_bm_free_queue": (_i, [_p, _p, _i64]),
    "pa_bm_block_table": (_i, [_p, _i64, _p, _i64]),
    "pa_bm_batch_tables": (_i, [_p, _p, _i64, _p, _i64, _p]),
    "pa_bm_num_pending_copies": (_i64, [_p]),
    "pa_bm_take_copies": (_i64, [_p, _p, _i64]),
    "pa_bm_enable_prefix_caching": (_i, [_p]),
    "pa_bm_add_seq_cached": (_i, [_p, _i64, _p, _i64, _i64, ctypes.POINTER(_i64)]),
    "pa_bm_append_tokens": (_i, [_p, _i64, _p, _i64, _p]),
    "pa_bm_append_tokens_batch": (_i, [_p, _p, _p, _i64, _p, _p, _p]),
    "pa_bm_prefix_stats": (_i, [_p, ctypes.POINTER(_i64), ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
}
for _name, (_res, _args) in _sig.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class PAError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = lib.pa_status_string(status).decode()
        if status == 4:
            msg += f" (cudaError {lib.pa_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [status {status}]")
        self.status = status


def _check(status: int, what: str):
    if status != 0:
        raise PAError(status, what)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return PA_F32
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.float8_e4m3fn:
        return PA_FP8_E4M3
    raise TypeError(f"unsupported dtype {t.dtype} (float32, bfloat16 or float8_e4m3fn)")


def _dev(t: torch.Tensor, name: str, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return t.data_ptr()


def _stream(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _cache_geometry(k_cache: torch.Tensor, v_cache: torch.Tensor):
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype or k_cache.dim() != 4:
        raise ValueError("k_cache and v_cache must both be [num_blocks, block_size, num_kv_heads, head_dim]")
    return tuple(int(x) for x in k_cache.shape)


def kv_write(k, v, k_cache, v_cache, slot_mapping, stream=None):
    """pa_kv_write: k_cache[slot // B, slot % B] = k[t] (and v) for every slot >= 0."""
    NB, B, Hkv, D = _cache_geometry(k_cache, v_cache)
    T = int(k.shape[0])
    if tuple(k.shape) != (T, Hkv, D) or tuple(v.shape) != (T, Hkv, D) or k.dtype != k_cache.dtype or \
            v.dtype != k_cache.dtype:
        raise ValueError("k, v must be [num_tokens, num_kv_heads, head_dim] in the cache dtype")
    if tuple(slot_mapping.shape) != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    st = lib.pa_kv_write(_dev(k, "k"), _dev(v, "v"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                         _dev(slot_mapping, "slot_mapping", torch.int64), T, NB, B, Hkv, D,
                         _dtype_code(k_cache), _stream(stream, k_cache.device))
    _check(st, "pa_kv_write")


def copy_blocks(k_cache, v_cache, block_mapping, stream=None):
    """pa_copy_blocks: for each (src, dst) row of block_mapping [n, 2], cache[dst] = cache[src]."""
    NB, B, Hkv, D = _cache_geometry(k_cache, v_cache)
    if block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
        raise ValueError("block_mapping must be [num_pairs, 2]")
    n = int(block_mapping.shape[0])
    ptr = _dev(block_mapping, "block_mapping", torch.int64) if n > 0 else 0
    st = lib.pa_copy_blocks(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ptr, n, NB, B, Hkv, D,
                            _dtype_code(k_cache), _stream(stream, k_cache.device))
    _check(st, "pa_copy_blocks")


def _out(t: torch.Tensor) -> int:
    """An attention output: a CUDA tensor, or a pinned host tensor (the kernels store the
    rows through its unified address; they are on the host once the stream has synchronised)."""
    if not isinstance(t, torch.Tensor) or not t.is_contiguous():
        raise ValueError("out must be a contiguous tensor")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError("out must be a CUDA tensor or pinned host memory")
    return t.data_ptr()


def _pool_ptr(t: torch.Tensor, name: str) -> int:
    """A CUDA tensor, or a pinned host tensor (used through its unified address)."""
    if not isinstance(t, torch.Tensor) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    return t.data_ptr()


def swap_blocks(src_k, src_v, dst_k, dst_v, block_mapping, stream=None):
    """pa_swap_blocks: dst[d] = src[s] for each (s, d) row of block_mapping [n, 2], whole blocks,
    between two pools of one block geometry; either pool may be pinned host memory."""
    if src_k.shape[1:] != dst_k.shape[1:] or src_k.dtype != dst_k.dtype or src_k.shape != src_v.shape or \
            dst_k.shape != dst_v.shape or src_k.dim() != 4:
        raise ValueError("pools must be [num_blocks, block_size, num_kv_heads, head_dim] of one geometry and dtype")
    if block_mapping.dim() != 2 or block_mapping.shape[1] != 2 or block_mapping.dtype != torch.int64:
        raise ValueError("block_mapping must be int64 [num_pairs, 2]")
    n = int(block_mapping.shape[0])
    _, B, Hkv, D = (int(x) for x in src_k.shape)
    dev = src_k.device if src_k.is_cuda else dst_k.device
    st = lib.pa_swap_blocks(_pool_ptr(src_k, "src_k"), _pool_ptr(src_v, "src_v"), _pool_ptr(dst_k, "dst_k"),
                            _pool_ptr(dst_v, "dst_v"), _pool_ptr(block_mapping, "block_mapping") if n else None, n,
                            int(src_k.shape[0]), int(dst_k.shape[0]), B, Hkv, D, _dtype_code(src_k),
                            _stream(stream, dev))
    _check(st, "pa_swap_blocks")


def attention_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int) -> int:
    """pa_attention_workspace_size for the current device."""
    out = ctypes.c_size_t(0)
    _check(lib.pa_attention_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, ctypes.byref(out)),
           "pa_attention_workspace_size")
    return int(out.value)


def attention(out, q, k_cache, v_cache, block_table, seq_lens, query_start_loc, *, max_query_len: int,
              max_seq_len: int, scale: float, workspace=None, stream=None):
    """pa_attention: paged decode + chunked-prefill attention of one varlen batch.

    out, q: [num_tokens, num_heads, head_dim]; block_table int32 [num_seqs, max_blocks];
    seq_lens int32 [num_seqs]; query_start_loc int32 [num_seqs + 1]. ``max_query_len`` and
    ``max_seq_len`` are host-side upper bounds. ``workspace`` is a uint8 CUDA tensor of at
    least attention_workspace_size(...) bytes (no initial contents needed); when None one is
    allocated with torch. ``out`` may be a pinned host tensor: the kernels then store the
    rows over the CPU-GPU link, and they are in place once the stream has synchronised.
    For a decode-only batch (max_query_len <= 1) ``q`` may be a pinned host tensor too: the
    decode kernel reads its rows over the link (no separate copy).
    """
    NB, B, Hkv, D = _cache_geometry(k_cache, v_cache)
    T, Hq = int(q.shape[0]), int(q.shape[1])
    if q.dim() != 3 or tuple(out.shape) != tuple(q.shape) or int(q.shape[2]) != D:
        raise ValueError("q and out must be [num_tokens, num_heads, head_dim]")
    if q.dtype != k_cache.dtype or out.dtype != k_cache.dtype:
        raise TypeError("q, out and the caches must share one dtype")
    S = int(seq_lens.shape[0])
    if block_table.dim() != 2 or int(block_table.shape[0]) != S or tuple(query_start_loc.shape) != (S + 1,):
        raise ValueError("block_table [S, W], seq_lens [S], query_start_loc [S + 1]")
    if workspace is None:
        workspace = torch.empty(attention_workspace_size(S, Hq, Hkv, D), dtype=torch.uint8, device=k_cache.device)
    ws_ptr = workspace.data_ptr() if workspace.numel() > 0 else 0
    st = lib.pa_attention(_out(out), _pool_ptr(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                          _dev(block_table, "block_table", torch.int32, 2), int(block_table.shape[1]),
                          _dev(seq_lens, "seq_lens", torch.int32, 1),
                          _dev(query_start_loc, "query_start_loc", torch.int32, 1), S, T, int(max_query_len),
                          int(max_seq_len), Hq, Hkv, D, B, NB, float(scale), _dtype_code(q), ws_ptr,
                          workspace.numel(), _stream(stream, k_cache.device))
    _check(st, "pa_attention")
    return out


def attention_fixed_scratch(out, q, k_cache, v_cache, block_table, seq_lens, query_start_loc, *,
                            max_query_len: int, max_seq_len: int, scale: float, stream=None):
    """pa_attention_fixed_scratch: attention() with the library's fixed scratch instead of a
    workspace, every kernel on ``stream`` (a batch with prefill rows runs one prefill launch
    over all SMs after the decode kernels). Calls that may overlap on the GPU race on the
    shared scratch."""
    NB, B, Hkv, D = _cache_geometry(k_cache, v_cache)
    T, Hq = int(q.shape[0]), int(q.shape[1])
    if q.dim() != 3 or tuple(out.shape) != tuple(q.shape) or int(q.shape[2]) != D:
        raise ValueError("q and out must be [num_tokens, num_heads, head_dim]")
    if q.dtype != k_cache.dtype or out.dtype != k_cache.dtype:
        raise TypeError("q, out and the caches must share one dtype")
    S = int(seq_lens.shape[0])
    if block_table.dim() != 2 or int(block_table.shape[0]) != S or tuple(query_start_loc.shape) != (S + 1,):
        raise ValueError("block_table [S, W], seq_lens [S], query_start_loc [S + 1]")
    st = lib.pa_attention_fixed_scratch(_out(out), _pool_ptr(q, "q"), _dev(k_cache, "k_cache"),
                                        _dev(v_cache, "v_cache"), _dev(block_table, "block_table", torch.int32, 2),
                                        int(block_table.shape[1]), _dev(seq_lens, "seq_lens", torch.int32, 1),
                                        _dev(query_start_loc, "query_start_loc", torch.int32, 1), S, T,
                                        int(max_query_len), int(max_seq_len), Hq, Hkv, D, B, NB, float(scale),
                                        _dtype_code(q), _stream(stream, k_cache.device))
    _check(st, "pa_attention_fixed_scratch")
    return out


def write_attention(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_table, seq_lens,
                    query_start_loc, *, max_query_len: int, max_seq_len: int, scale: float, workspace=None,
                    stream=None):
    """pa_write_attention: kv_write(k_new, v_new, ..., slot_mapping) then attention(...), in one call.

    For a decode request (q_len 1, length L) slot_mapping of its token must be the slot of
    position L - 1 in its block table; the decode kernel then writes it itself. For a
    decode-only batch, q, k_new and v_new may be pinned host tensors (read over the link).
    """
    NB, B, Hkv, D = _cache_geometry(k_cache, v_cache)
    T, Hq = int(q.shape[0]), int(q.shape[1])
    if q.dim() != 3 or tuple(out.shape) != tuple(q.shape) or int(q.shape[2]) != D:
        raise ValueError("q and out must be [num_tokens, num_heads, head_dim]")
    if q.dtype != k_cache.dtype or out.dtype != k_cache.dtype:
        raise TypeError("q, out and the caches must share one dtype")
    if tuple(k_new.shape) != (T, Hkv, D) or tuple(v_new.shape) != (T, Hkv, D) or \
            k_new.dtype != k_cache.dtype or v_new.dtype != k_cache.dtype:
        raise ValueError("k_new, v_new must be [num_tokens, num_kv_heads, head_dim] in the cache dtype")
    if tuple(slot_mapping.shape) != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    S = int(seq_lens.shape[0])
    if block_table.dim() != 2 or int(block_table.shape[0]) != S or tuple(query_start_loc.shape) != (S + 1,):
        raise ValueError("block_table [S, W], seq_lens [S], query_start_loc [S + 1]")
    if workspace is None:
        workspace = torch.empty(attention_workspace_size(S, Hq, Hkv, D), dtype=torch.uint8, device=k_cache.device)
    ws_ptr = workspace.data_ptr() if workspace.numel() > 0 else 0
    st = lib.pa_write_attention(_out(out), _pool_ptr(q, "q"), _pool_ptr(k_new, "k_new"), _pool_ptr(v_new, "v_new"),
                                _dev(slot_mapping, "slot_mapping", torch.int64), _dev(k_cache, "k_cache"),
                                _dev(v_cache, "v_cache"), _dev(block_table, "block_table", torch.int32, 2),
                                int(block_table.shape[1]), _dev(seq_lens, "seq_lens", torch.int32, 1),
                                _dev(query_start_loc, "query_start_loc", torch.int32, 1), S, T, int(max_query_len),
                                int(max_seq_len), Hq, Hkv, D, B, NB, float(scale), _dtype_code(q), ws_ptr,
                                workspace.numel(), _stream(stream, k_cache.device))
    _check(st, "pa_write_attention")
    return out


def kv_write_fp8(k, v, k_cache, v_cache, slot_mapping, k_scale: float, v_scale: float, stream=None):
    """pa_kv_write_fp8: cache[slot] = E4M3(x / scale) for every slot >= 0; k, v bf16 or
    float32 [num_tokens, num_kv_heads, head_dim]; caches torch.float8_e4m3fn."""
    NB, B, Hkv, D = _cache_geometry(k_cache, v_cache)
    if k_cache.dtype != torch.float8_e4m3fn:
        raise TypeError("the caches must be torch.float8_e4m3fn")
    T = int(k.shape[0])
    if tuple(k.shape) != (T, Hkv, D) or tuple(v.shape) != (T, Hkv, D) or k.dtype != v.dtype:
        raise ValueError("k, v must be [num_tokens, num_kv_heads, head_dim] of one dtype")
    if tuple(slot_mapping.shape) != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    st = lib.pa_kv_write_fp8(_dev(k, "k"), _dev(v, "v"), _dtype_code(k), _dev(k_cache, "k_cache"),
                             _dev(v_cache, "v_cache"), _dev(slot_mapping, "slot_mapping", torch.int64), T, NB, B,
                             Hkv, D, float(k_scale), float(v_scale), _stream(stream, k_cache.device))
    _check(st, "pa_kv_write_fp8")


def attention_fp8(out, q, k_cache, v_cache, block_table, seq_lens, query_start_loc, *, max_query_len: int,
                  max_seq_len: int, scale: float, k_scale: float, v_scale: float, workspace=None, stream=None):
    """pa_attention_fp8: attention() over float8_e4m3fn caches (values = code * scale);
    q and out bfloat16."""
    NB, B, Hkv, D = _cache_geometry(k_cache, v_cache)
    if k_cache.dtype != torch.float8_e4m3fn:
        raise TypeError("the caches must be torch.float8_e4m3fn")
    T, Hq = int(q.shape[0]), int(q.shape[1])
    if q.dim() != 3 or tuple(out.shape) != tuple(q.shape) or int(q.shape[2]) != D:
        raise ValueError("q and out must be [num_tokens, num_heads, head_dim]")
    if q.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise TypeError("q and out must be bfloat16")
    S = int(seq_lens.shape[0])
    if block_table.dim() != 2 or int(block_table.shape[0]) != S or tuple(query_start_loc.shape) != (S + 1,):
        raise ValueError("block_table [S, W], seq_lens [S], query_start_loc [S + 1]")
    if workspace is None:
        workspace = torch.empty(attention_workspace_size(S, Hq, Hkv, D), dtype=torch.uint8, device=k_cache.device)
    ws_ptr = workspace.data_ptr() if workspace.numel() > 0 else 0
    st = lib.pa_attention_fp8(_out(out), _pool_ptr(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                              _dev(block_table, "block_table", torch.int32, 2), int(block_table.shape[1]),
                              _dev(seq_lens, "seq_lens", torch.int32, 1),
                              _dev(query_start_loc, "query_start_loc", torch.int32, 1), S, T, int(max_query_len),
                              int(max_seq_len), Hq, Hkv, D, B, NB, float(scale), float(k_scale), float(v_scale),
                              ws_ptr, workspace.numel(), _stream(stream, k_cache.device))
    _check(st, "pa_attention_fp8")
    return out


def attention_grouped_workspace_size(num_seqs: int, num_groups: int, num_heads: int, num_kv_heads: int,
                                     head_dim: int) -> int:
    """pa_attention_grouped_workspace_size for the current device."""
    out = ctypes.c_size_t(0)
    _check(lib.pa_attention_grouped_workspace_size(num_seqs, num_groups, num_heads, num_kv_heads, head_dim,
                                                   ctypes.byref(out)), "pa_attention_grouped_workspace_size")
    return int(out.value)


def attention_grouped(out, q, k_cache, v_cache, block_table, seq_lens, query_start_loc, seq_group, group_range,
                      shared_len, *, max_seq_len: int, scale: float, workspace=None, stream=None):
    """pa_attention_grouped: decode attention where each group's shared prefix is read once.

    seq_group int32 [S], group_range int32 [num_groups, 2], shared_len int32 [num_groups]
    (from BlockManager.batch_groups); the result equals attention() on the same batch."""
    NB, B, Hkv, D = _cache_geometry(k_cache, v_cache)
    T, Hq = int(q.shape[0]), int(q.shape[1])
    if q.dim() != 3 or tuple(out.shape) != tuple(q.shape) or int(q.shape[2]) != D:
        raise ValueError("q and out must be [num_tokens, num_heads, head_dim]")
    S = int(seq_lens.shape[0])
    G = int(shared_len.shape[0])
    if tuple(seq_group.shape) != (S,) or tuple(group_range.shape) != (G, 2):
        raise ValueError("seq_group [S], group_range [num_groups, 2], shared_len [num_groups]")
    if workspace is None:
        workspace = torch.empty(attention_grouped_workspace_size(S, G, Hq, Hkv, D), dtype=torch.uint8,
                                device=k_cache.device)
    grp = lambda t, n: _dev(t, n, torch.int32) if G > 0 else 0  # noqa: E731
    st = lib.pa_attention_grouped(_out(out), _pool_ptr(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                                  _dev(block_table, "block_table", torch.int32, 2), int(block_table.shape[1]),
                                  _dev(seq_lens, "seq_lens", torch.int32, 1),
                                  _dev(query_start_loc, "query_start_loc", torch.int32, 1), S, T, int(max_seq_len),
                                  Hq, Hkv, D, B, NB, float(scale), _dtype_code(q), grp(seq_group, "seq_group"),
                                  grp(group_range, "group_range"), grp(shared_len, "shared_len"), G,
                                  workspace.data_ptr() if workspace.numel() else 0, workspace.numel(),
                                  _stream(stream, k_cache.device))
    _check(st, "pa_attention_grouped")
    return out


def read_device_errors(clear: bool = True) -> int:
    """The current device's error word (PA_DEVERR bits); synchronises the device."""
    flags = ctypes.c_uint(0)
    _check(lib.pa_read_device_errors(ctypes.byref(flags), 1 if clear else 0), "pa_read_device_errors")
    return int(flags.value)


class BlockManager:
    """pa_bm_*: host block accounting (free queue, tables, ref counts, copy-on-write)."""

    def __init__(self, num_blocks: int, block_size: int, free_order):
        import numpy as np

        order = np.ascontiguousarray(np.asarray(free_order, dtype=np.int32))
        if order.shape != (num_blocks,):
            raise ValueError("free_order must have num_blocks entries")
        self._h = lib.pa_bm_create(num_blocks, block_size, order.ctypes.data)
        if not self._h:
            raise ValueError("pa_bm_create: free_order must be a permutation of range(num_blocks)")
        self.num_blocks, self.block_size = num_blocks, block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib.pa_bm_destroy(h)
            self._h = None

    def add_seq(self, seq: int):
        _check(lib.pa_bm_add_seq(self._h, seq), "pa_bm_add_seq")

    def append(self, seq: int, n: int):
        """Returns the slots of the n new tokens (numpy int64)."""
        import numpy as np

        out = np.empty(max(n, 0), np.int64)
        _check(lib.pa_bm_append(self._h, seq, n, out.ctypes.data if n > 0 else None), "pa_bm_append")
        return out

    def append_batch(self, seqs, counts, out=None):
        """Append counts[i] tokens to seqs[i] for every i (one C call); returns the slots,
        concatenated (numpy int64). ``out`` may be a preallocated int64 array."""
        import numpy as np

        s = np.ascontiguousarray(np.asarray(seqs, np.int64))
        c = np.ascontiguousarray(np.asarray(counts, np.int64))
        total = int(c.sum())
        if out is None:
            out = np.empty(total, np.int64)
        elif out.dtype != np.int64 or not out.flags.c_contiguous or out.size < total:
            raise ValueError("out must be a contiguous int64 array of at least sum(counts) entries")
        done = ctypes.c_int64(0)
        st = lib.pa_bm_append_batch(self._h, s.ctypes.data if len(s) else None, c.ctypes.data if len(c) else None,
                                    len(s), out.ctypes.data if total else None, ctypes.byref(done))
        _check(st, f"pa_bm_append_batch (stopped after {done.value} entries)")
        return out[:total]

    # -- prefix caching ----------------------------------------------------------
    def enable_prefix_caching(self):
        _check(lib.pa_bm_enable_prefix_caching(self._h), "pa_bm_enable_prefix_caching")

    def add_seq_cached(self, seq: int, prompt, max_hit: int) -> int:
        """Start ``seq`` from the longest cached prefix of ``prompt`` (token ids); returns
        the number of tokens reused."""
        import numpy as np

        t = np.ascontiguousarray(np.asarray(prompt, np.int32))
        hit = ctypes.c_int64(0)
        _check(lib.pa_bm_add_seq_cached(self._h, seq, t.ctypes.data if t.size else None, t.size, max_hit,
                                        ctypes.byref(hit)), "pa_bm_add_seq_cached")
        return int(hit.value)

    def append_tokens(self, seq: int, tokens):
        """Append the tokens ``tokens`` (ids) to ``seq``; returns their slots (numpy int64)."""
        import numpy as np

        t = np.ascontiguousarray(np.asarray(tokens, np.int32))
        out = np.empty(t.size, np.int64)
        _check(lib.pa_bm_append_tokens(self._h, seq, t.ctypes.data if t.size else None, t.size,
                                       out.ctypes.data if t.size else None), "pa_bm_append_tokens")
        return out

    def append_tokens_batch(self, seqs, counts, tokens, out=None):
        """append_batch with token ids (``tokens`` concatenated in entry order)."""
        import numpy as np

        s = np.ascontiguousarray(np.asarray(seqs, np.int64))
        c = np.ascontiguousarray(np.asarray(counts, np.int64))
        t = np.ascontiguousarray(np.asarray(tokens, np.int32))
        total = int(c.sum())
        if t.size < total:
            raise ValueError("tokens must hold sum(counts) ids")
        if out is None:
            out = np.empty(total, np.int64)
        elif out.dtype != np.int64 or not out.flags.c_contiguous or out.size < total:
            raise ValueError("out must be a contiguous int64 array of at least sum(counts) entries")
        done = ctypes.c_int64(0)
        st = lib.pa_bm_append_tokens_batch(self._h, s.ctypes.data if len(s) else None,
                                           c.ctypes.data if len(c) else None, len(s),
                                           t.ctypes.data if total else None, out.ctypes.data if total else None,
                                           ctypes.byref(done))
        _check(st, f"pa_bm_append_tokens_batch (stopped after {done.value} entries)")
        return out[:total]

    def prefix_stats(self):
        """(registered blocks, blocks reused by lookups, registrations evicted)."""
        a, b, c = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
        _check(lib.pa_bm_prefix_stats(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
               "pa_bm_prefix_stats")
        return int(a.value), int(b.value), int(c.value)

    def batch_groups(self, seqs, max_members: int):
        """(seq_group int32 [n], group_range int32 [groups, 2], shared_len int32 [groups]) for
        pa_attention_grouped over the batch ``seqs`` (batch order)."""
        import numpy as np

        s = np.ascontiguousarray(np.asarray(seqs, np.int64))
        n = len(s)
        cap = max(n // 2, 1)
        sg = np.empty(n, np.int32)
        gr = np.empty((cap, 2), np.int32)
        sl = np.empty(cap, np.int32)
        ng = ctypes.c_int64(0)
        _check(lib.pa_bm_batch_groups(self._h, s.ctypes.data if n else None, n, max_members,
                                      sg.ctypes.data if n else None, gr.ctypes.data, sl.ctypes.data, cap,
                                      ctypes.byref(ng)), "pa_bm_batch_groups")
        return sg, gr[: ng.value].copy(), sl[: ng.value].copy()

    # -- swapping ----------------------------------------------------------------
    def enable_swap(self, num_cpu_blocks: int, cpu_free_order):
        import numpy as np

        order = np.ascontiguousarray(np.asarray(cpu_free_order, dtype=np.int32))
        if order.shape != (num_cpu_blocks,):
            raise ValueError("cpu_free_order must have num_cpu_blocks entries")
        _check(lib.pa_bm_enable_swap(self._h, num_cpu_blocks, order.ctypes.data), "pa_bm_enable_swap")

    def _swap(self, fn, what, seqs):
        import numpy as np

        s = np.ascontiguousarray(np.asarray(seqs, np.int64))
        cap = sum(int(lib.pa_bm_num_seq_blocks(self._h, int(x))) for x in s)
        out = np.empty((max(cap, 1), 2), np.int64)
        n = ctypes.c_int64(0)
        _check(fn(self._h, s.ctypes.data if len(s) else None, len(s), out.ctypes.data, cap, ctypes.byref(n)), what)
        return out[: n.value]

    def swap_out(self, seqs):
        """Move the group to the CPU pool; returns the (gpu, cpu) pairs to copy, int64 [n, 2]."""
        return self._swap(lib.pa_bm_swap_out, "pa_bm_swap_out", seqs)

    def swap_in(self, seqs):
        """Move the group back to the GPU; returns the (cpu, gpu) pairs to copy, int64 [n, 2]."""
        return self._swap(lib.pa_bm_swap_in, "pa_bm_swap_in", seqs)

    def is_swapped(self, seq: int) -> bool:
        r = int(lib.pa_bm_is_swapped(self._h, seq))
        if r < 0:
            raise PAError(7, "pa_bm_is_swapped")
        return bool(r)

    def num_free_cpu(self) -> int:
        return int(lib.pa_bm_num_free_cpu(self._h))

    def cpu_ref_count(self, block: int) -> int:
        return int(lib.pa_bm_cpu_ref_count(self._h, block))

    def fork(self, parent: int, child: int):
        _check(lib.pa_bm_fork(self._h, parent, child), "pa_bm_fork")

    def free_seq(self, seq: int):
        _check(lib.pa_bm_free_seq(self._h, seq), "pa_bm_free_seq")

    def seq_len(self, seq: int) -> int:
        return int(lib.pa_bm_seq_len(self._h, seq))

    def ref_count(self, block: int) -> int:
        return int(lib.pa_bm_ref_count(self._h, block))

    def num_free(self) -> int:
        return int(lib.pa_bm_num_free(self._h))

    def free_queue(self):
        import numpy as np

        out = np.empty(self.num_free(), np.int32)
        _check(lib.pa_bm_free_queue(self._h, out.ctypes.data if out.size else None, out.size), "pa_bm_free_queue")
        return out

    def block_table(self, seq: int):
        import numpy as np

        n = int(lib.pa_bm_num_seq_blocks(self._h, seq))
        if n < 0:
            raise PAError(7, "pa_bm_block_table")
        out = np.empty(n, np.int32)
        _check(lib.pa_bm_block_table(self._h, seq, out.ctypes.data if n else None, n), "pa_bm_block_table")
        return out

    def batch_tables(self, seqs, width: int, table_out=None, lens_out=None):
        """(block_table int32 [n, width], seq_lens int32 [n]) for the sequences ``seqs``,
        written into ``table_out`` / ``lens_out`` when given (contiguous int32 arrays)."""
        import numpy as np

        s = np.ascontiguousarray(np.asarray(seqs, np.int64))
        table = np.empty((len(s), width), np.int32) if table_out is None else table_out
        lens = np.empty(len(s), np.int32) if lens_out is None else lens_out
        if table.shape != (len(s), width) or lens.shape != (len(s),) or table.dtype != np.int32 or \
                lens.dtype != np.int32 or not table.flags.c_contiguous or not lens.flags.c_contiguous:
            raise ValueError("table_out must be int32 [n, width] and lens_out int32 [n], contiguous")
        _check(lib.pa_bm_batch_tables(self._h, s.ctypes.data if len(s) else None, len(s),
                                      table.ctypes.data if len(s) else None, width,
                                      lens.ctypes.data if len(s) else None), "pa_bm_batch_tables")
        return table, lens

    def take_copies(self):
        """Pending copy-on-write pairs, oldest first: int64 [n, 2] (src, dst)."""
        import numpy as np

        n = int(lib.pa_bm_num_pending_copies(self._h))
        out = np.empty((n, 2), np.int64)
        got = lib.pa_bm_take_copies(self._h, out.ctypes.data if n else None, n)
        if got != n:
            raise PAError(1, "pa_bm_take_copies")
        return out
