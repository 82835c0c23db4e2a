"""CPU float64 oracle for GQA decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never calls it and has no fallback to it.

Every function is written from the method's definition on the pages:

* page "kernbench2 ... _gqa_attention_decode_long.py" ("GQA fused-attention
  decode kernel -- long context"): the tensor layout in the kernel docstring,
  the local attention of one S_kv tile (scores, row max, exp, row sum, exp@V),
  ``_merge_running`` (the online-softmax merge of two (m, l, O) partials) and
  the final normalise ``O / l`` at the root;
* page "project_6 ... muh_kernel_map.py", ``VLLM_KERNEL_MAP`` rows
  ``paged_attention_v1`` / ``paged_attention_v2``: fp32 scores, fp16 output,
  the paged KV cache and the two-pass partitioned reduce + merge.

All arithmetic is float64 on exact float16 inputs (float16 -> float64 is exact).
Pins (brute force, closed forms, library special cases, invariants) are in
``tests/test_oracle_pins.py``; every function here is pinned.
"""
from .gqa_oracle import (  # noqa: F401
    partial_rows,
    merge_pair,
    merge_parts,
    normalize,
    decode,
    decode_unit,
    decode_partial,
    gather_paged,
    gather_paged_vllm,
    decode_paged,
    decode_paged_seq,
)

__all__ = [
    "partial_rows", "merge_pair", "merge_parts", "normalize", "decode", "decode_unit",
    "decode_partial", "gather_paged", "gather_paged_vllm", "decode_paged", "decode_paged_seq",
]
