"""CPU oracle for the CacheBlend blend step -- TEST INFRASTRUCTURE ONLY.

Plain, slow, float64 numpy code written from the CacheBlend deep-dive page.
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import it; the CUDA library never does, and the two share no
code (the seeded input generator in ``workload/`` is their only common input).

Every function is pinned by a CPU test against something other than itself
(closed forms, invariants of the method, a brute-force sequential decoder,
library routines for special cases, and the page's printed sizing numbers).
The selected set at 0 < r < 1 has no printed worked example on the pages; it is
pinned only through the page's Δkv definition against a brute-force full prefill.
"""
from .cpu_blend import (attention, blend, blend_gradual, chunk_caches, deviation, deviation_rows, gradual_counts, prefill,
                        rerope, rmsnorm, rope, rope_freqs, round_bf16, round_store, select_hkvd, selected_count, silu,
                        to_f64, Model, validate_chunks)
from . import accounting
from . import matcher

__all__ = ["attention", "blend", "blend_gradual", "gradual_counts", "chunk_caches", "deviation", "deviation_rows", "prefill", "rerope", "rmsnorm", "rope",
           "rope_freqs", "round_bf16", "round_store", "select_hkvd", "selected_count", "silu", "to_f64",
           "Model", "validate_chunks", "accounting", "matcher"]
