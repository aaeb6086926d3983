"""Seeded synthetic inputs for the paged-attention hot path.

This module is shared by the float64 oracle and by the CUDA path. It holds none
of the method's arithmetic: it only fixes shapes, lengths, pool sizes, the
permutation in which physical block ids are handed out, a script of block-manager
operations (add a sequence, append tokens, fork, admit a prompt, end a request),
token ids where prefix caching needs them, and the random values of q / K / V. Everything the method computes from these (slot mappings, block
tables, CoW pairs, cache contents, attention outputs) is computed separately
by each side.

Values are drawn per append operation from a NumPy PCG64 stream keyed by
(seed, kind, sequence, start position), so any subset of sequences can be
regenerated without drawing the rest.
"""
from .configs import (  # noqa: F401
    CONFIGS,
    Phase,
    Spec,
    Workload,
    build,
    custom,
    relevant_seqs,
    preemption,
    shared_prefix,
    system_prompt,
    with_fp8_cache,
)
