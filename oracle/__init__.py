"""CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 restatement of what the hot path computes, written from
the pages' definitions and independent of the CUDA library: it shares no
code, header, table or constant with ``paged_kv_cache_254_gb300`` and neither
imports the other.  Only the test suite, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The product path never routes through here.

Sources (the three pages on PagedAttention):
  * "AI Inference Serving at Scale ..." (ontq.xyz), section 3 "PagedAttention:
    Virtual Memory and Paging for GPU Tensors" -- block pool, block table,
    on-demand allocation, copy-on-write; section 8 FAQ -- paged attention is
    identical to un-paged attention; section 2 -- KV bytes per token.
  * "How LLM Inference Engines Work ..." (letsbuildsolutions.com), section
    "PagedAttention: Virtual Memory for KV Caches" -- the BlockManager sketch
    (LIFO free list, refcount, allocate/free) and the gather requirement;
    section "KV Caches" -- per-layer KV bytes.
  * "vLLM & High-Throughput Serving ..." (thewebvale.com), section 2 "The
    Block Table" -- logical block i = floor(t / B), offset j = t mod B;
    section 1 -- Llama-3-70B KV bytes per token.

Every function here is pinned by ``tests/test_oracle*.py`` to something other
than itself: closed forms, brute force on tiny inputs, the pages' worked
numbers (``tests/golden/``), invariants.  Nothing is "parity unpinned".
"""
