"""Oracle: a plain, slow, float64 CPU statement of the paged-attention hot path.

TEST INFRASTRUCTURE ONLY. It exists to check the CUDA library, and only the
tests, the smoke check and the benchmark's CPU-baseline leg may import it. It
shares no code with the CUDA path: not a kernel, a header, a helper, a table
or a constant generator. The seeded inputs both sides consume come from the
separate ``workloads`` package, which holds none of the method's arithmetic.

Contents, each citing the page passage it follows:
- block_manager.BlockAllocator: blocks, tables, ref counts, fork, copy-on-write.
- prefix_cache.PrefixCachingAllocator: the same plus reuse of cached full blocks
  found by their token prefix, with LRU eviction through the free queue.
- fp8: the E4M3 cache format, quantised writes (kv_write_fp8_ref) and dequantisation.
- swap.SwappingAllocator / SwappingPrefixAllocator: a CPU block pool and the swap out /
  swap in of preempted sequence groups.
- attention.kv_write_ref / copy_blocks_ref / paged_attention_ref /
  dense_causal_ref: the byte moves and the float64 attention.
- runner.run_workload: a seeded workload, phase by phase.

Every function is pinned by the CPU tests (the pages' worked examples, closed
forms, invariants, brute force and a library cross-check); none is unpinned.
"""
from .attention import (  # noqa: F401
    BlockStore,
    attend,
    copy_blocks_ref,
    dense_causal_ref,
    gather_kv,
    kv_write_ref,
    paged_attention_ref,
    to_f64,
)
from .block_manager import BlockAllocator, NoFreeBlocks, TooLarge  # noqa: F401
from .prefix_cache import PrefixCachingAllocator  # noqa: F401
from .fp8 import dequantize, kv_write_fp8_ref, quantize  # noqa: F401
from .swap import SwappingAllocator, SwappingPrefixAllocator  # noqa: F401
from .runner import (OracleResult, batch_metadata, run_allocator, run_script, run_script_swaps,  # noqa: F401
                     run_workload, step_ranges)
