"""FP64 CPU oracle for paged GQA decode and fused RoPE + paged KV append.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may call it.  It shares no code with the CUDA library; its only
common dependency is the seeded input module ``workloads``.

It is a plain restatement of what the hot path computes, written for a reader
to check by eye, in FP64 NumPy with per-element loops where that is clearer:

* ``bf16``       bf16 <-> float conversions (widening is exact; narrowing is
                 round-to-nearest-even).
* ``rope``       RoPE frequencies, the fp32 cos/sin table, and the rotation in
                 the fixed fp32 operation order that makes the append bit-exact.
* ``paged_kv``   append into 16-token pages through per-sequence block tables,
                 and decode attention over a sequence's own pages (the softmax
                 definition, plus a split/log-sum-exp-combine restatement).
* ``int8_kv``    INT8 K/V pages: per-row symmetric 8-bit codes with fp32
                 scales, the quantised append, and decode over the
                 dequantised pages.
* ``argmax``     next-token selection over FP32 logits (first index of the
                 largest non-NaN value).
* ``admission``  the admission-credit rule and a FIFO continuous-batching
                 simulation with on-demand page allocation.

Sources (titles of the pages that define the path):
  - samir-vllm article (techfi24, "samir-vllm implemente l'inference Llama 3.2
    1B en C++/CUDA"), sections "Architecture et flux d'inference" (GQA, RoPE,
    BF16 storage, FP32 reductions) and "Gestion de la KV cache et strategies
    de batching" (16-token pages, per-sequence per-layer block tables, append at
    the absolute RoPE position, paged attention over the sequence's own pages,
    admission credit, rejection of oversize requests).
  - "Lifecycle and Memory Model" (TinyLoop C++ API), section "Per-request /
    handle-owned memory" (a request's KV cache stored as FP16 or INT8 K/V).
  - tiny-vllm chapter "2. Weight Loading and GPU Buffer Design", sections
    "Preallocating the 16 compute buffers" (model constants) and "What else is
    set up in the initialization block" (block table initialised to -1).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, invariants, brute force, library routines); none is unpinned.
"""
from . import admission, argmax, bf16, int8_kv, paged_kv, rope  # noqa: F401
