"""Plain, slow fp64 CPU oracle for prefix-shared decode attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import anything here; the
library's product path never does and shares no code with it.

What it computes (sources are named by page title and section):

* ``attention``  -- the definition softmax(q K^T / sqrt(d)) V over each
  sequence's full, unshared K/V (Cost-Efficient LLM Serving for Multi-turn
  Conversations with CachedAttention, "Load-bearing equations"; ChunkAttention,
  Knowl 3), and causal chunked prefill (Chunked Prefill, sections 1 and 2).
* ``tpp``        -- the two-phase partition algorithm step by step: partial_attn,
  attn_reduce and the final divide (ChunkAttention, Knowls 2 and 3).
* ``tree``       -- an independent prefix-tree model: prefix match, insert,
  append, remove, depth-first batch order and the canonical chunk tables
  (ChunkAttention, Knowls 1 and 5).
* ``schedule``   -- the W-row block split of a prompt (Chunked Prefill, section 3).
* ``theory``     -- sharing ratio, capacity multiplier and fragmentation bound
  (ChunkAttention, Knowl 4).

Every function is pinned by ``tests/test_oracle_*.py`` against library
routines, closed forms, worked examples printed on the pages, invariants and
brute force; nothing in it is marked "parity unpinned".
"""
