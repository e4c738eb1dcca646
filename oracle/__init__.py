"""CPU oracle for paged decode: plain, slow, obviously correct, fp64.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute anything in this package.  Only the test suite, the smoke check and
the benchmark's CPU-baseline leg use it.  It shares no code with the CUDA
path (``paged_kv_cache_216_gb300``) and imports nothing from it; the one
module both sides use is the seeded input generator ``workloads``.

Sources (web pages on paged KV caches):
  * "Day 6/90 of Inference Engineering" (bittide.aicompass.dev post, its
    notes on PagedAttention, paragraphs 2, 5 and 6): the KV cache manager
    hands out one fixed-size cache block at a time and takes a new one when
    the last is full; sequences with a common prefix share its blocks and
    write to a fresh block from the token where they diverge; a block table
    makes the scattered blocks read like one contiguous KV sequence.
  * "PagedAttention Kernel：大模型推理优化的显存管理革新" (intelliparadigm.com),
    section 3.1: attention over the paged cache is Q·Kᵀ block by block, a
    softmax, then P·V block by block.

Modules:
  attention  decode output by the plain definition softmax(scale·q·Kᵀ)·V
  cache      KV append (scatter into slots, also into an FP8 cache) and block copy
  fp8        E4M3 codes: quantize with a scale, decode
  prefill    append a prompt's tokens, then causal attention of each of them
  allocator  block allocator: free list, ref-counted sharing, copy-on-write
  serving    the serving loop (allocate, append, decode) built from the above

Every function is pinned by tests in ``tests/test_oracle*.py`` against
values fixed by the mathematics (closed forms, special cases, invariances,
library routines on contiguous data) and by hand-derived fixtures in
``tests/golden/``.
"""
