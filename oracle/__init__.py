"""Float64 CPU oracle for paged, causal, GQA prefill attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
library (``invariant_paged_prefill_gb300``) and imports nothing from it.

Contents
--------
``formats``          bit-level decoders for bf16 and OCP FP8 E4M3 storage.
``paged_attention``  the definition of tail-aligned causal GQA attention over
                     a paged KV cache, in float64.
"""

from .formats import bf16_bits_to_f64, e4m3_bits_to_f64
from .paged_attention import (
    kv_head_of,
    kv_lengths,
    paged_prefill,
    q_lengths,
    row_position,
)

__all__ = [
    "bf16_bits_to_f64",
    "e4m3_bits_to_f64",
    "kv_head_of",
    "kv_lengths",
    "paged_prefill",
    "q_lengths",
    "row_position",
]
