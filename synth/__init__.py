"""Seeded synthetic inputs shared by the oracle's tests and the CUDA path's
tests and benchmark.

This module holds no arithmetic of the method itself (no addressing, no
softmax, no block accounting).  It only fixes shapes, seeds, value
distributions and the order of block-manager operations that build each
workload; each side (oracle or CUDA library) executes those operations with
its own code.

Values: q, K and V are drawn as float32 N(0, 1) from NumPy's PCG64 generator
seeded per use, then stored either as float32 or rounded to bfloat16
(round-to-nearest-even, via torch's CPU conversion) and kept as raw uint16
bit patterns, so that the oracle and the GPU receive identical bits.
"""

from __future__ import annotations

from .workloads import (  # noqa: F401
    WORKLOADS,
    PrefillWorkload,
    Workload,
    normal_f32,
    storage_values,
    storage_dtype,
    permutation,
    recipe_lengths,
    restrict,
    workload,
    torch_seed,
)
