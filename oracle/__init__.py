"""Float64 CPU oracle for the agentic KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call,
link or execute this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code with the CUDA path (``agentic_kv_cache_gb300``): no
kernels, headers, helpers, tables or constant generators.  The one thing both
sides consume is the seeded input generator ``agentic_kv_cache_gb300.synth``,
which holds none of the method's arithmetic.

Sources (web pages, cited by title and section):

* [AKV-blog]  "AKV: Cache Engineering for Autonomous Agents and
  State-Preserving Prefix Invalidation Bypass" (Abrar Akhunji).
* [AKV-notes] "Cache Engineering for Agents" (reading notes on Fu et al.).
* [Leyline]   "Leyline: KV Cache Directives for Agentic Inference" (digest).

Modules
-------
bf16       round-to-nearest-even float64 -> bfloat16, bit patterns.
rope       RoPE angles, rotation, the repos primitive (k' = R(delta) k).
cache      the paged KV bookkeeping model: pages, sequences, fork/CoW,
           append / drop / repos / splice, flush run lists, segment run lists.
attention  masked softmax attention and segment-batch attention (bottom-right
           causal over a segment's visible KV list), with LSE.
kernels    what the GPU kernels compute, written as plain loops over the
           run lists the bookkeeping model produces (repos over paged pools,
           paged segment attention, compaction copies, attention mass).
radix      extended radix-tree matching (exact vs retrigger) by brute force
           over the inserted paths.

Every function here is pinned by a ``-m "not gpu"`` test against something
other than itself (closed forms, the pages' worked examples, library routines,
brute force); ``tests/test_oracle_*.py`` hold the pins.
"""
