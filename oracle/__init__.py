"""Oracle for paged decode attention, KV append and the block allocator.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

It is a plain, slow, obviously-correct CPU restatement of what the pages
describe, written in numpy with every floating-point result accumulated in
float64.  It shares no code with the CUDA library (no kernels, headers,
constants or helpers); the only thing both sides share is the seeded input
generator in ``synth/``, which holds none of the method's arithmetic.

Pages cited (by title and section):

* [VK]  vaibhawkumar.in, "Why LLMs run out of VRAM: KV cache fragmentation
        and the PagedAttention fix"
* [DEV] dev.to/syed_anzar, "Why LLMs Run Out of VRAM: KV Cache Fragmentation
        and How PagedAttention Fixes It"
* [HI]  hyperinfer.ai, "KV cache & paged attention deep dive"

Modules
-------
closed_forms  bytes per token, blocks per sequence, tail waste
e4m3          OCP FP8 E4M3 ("FN") decode / encode (RNE, saturate to +-448)
numerics      exact bf16 / f16 / f32 bit conversions used by the cache model
cache         slot mapping, KV append into the paged pool, logical gather
attention     single-query decode attention, contiguous and paged
split         split-context partitions and their log-sum-exp merge
allocator     physical block pool: LIFO free stack, refcounts, copy-on-write

Every function is pinned by ``tests/test_oracle_*.py`` against something
other than itself (values printed on the pages, closed forms, library
routines, brute force on tiny inputs).
"""
