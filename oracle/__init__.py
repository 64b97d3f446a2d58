"""Oracle for the paged decode path: plain, slow, fp64 CPU restatement.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import, call or execute anything under ``oracle/``.  It shares
no code, tables or helpers with the CUDA library in
``paged_kv_cache_228_gb300/csrc``; the only common dependency is the seeded
input generator module ``paged_kv_cache_228_gb300.workloads``, which holds none
of the method's arithmetic.

Modules
-------
paged_attention
    Cache write (scatter append), block copy (copy-on-write) and paged decode
    attention: gather each sequence's K/V through its block table into a
    contiguous fp64 array, then dense softmax(q K^T * scale) V.
e4m3
    OCP OFP8 E4M3 codec written from the format definition (decode table and a
    round-to-nearest-even, saturating fp32 -> E4M3 encoder).
quantize
    Per-(block, KV head) absmax FP8 quantisation of cache blocks.
e2m1
    FP4 E2M1 element codec from the OCP MX definition (decode table and a
    round-to-nearest-even, saturating encoder).
nvfp4
    Two-level scaled NVFP4 cache (E2M1 values, one E4M3 scale per 16 values,
    one fp32 scale per tensor): quantiser, byte layout, decode attention.
block_manager
    Dictionary/list model of the host block allocator (free list, refcounts,
    fork, copy-on-write append).
footprint
    Per-token KV footprint formula used for the algorithmic byte count.

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
invariants, brute force and library routines (see each test's docstring).
"""
