"""Oracle for prefix-shared tree decode attention -- TEST INFRASTRUCTURE.

A plain, slow, obviously correct CPU statement of what the tree decode path
computes, in fp64. It exists to check the CUDA path and nothing else: only the
tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may import
it; the product path never calls it and falls over loudly if its CUDA library
is missing.

It shares no code with the library: its own page walk, its own path walk, its
own bf16 decoding. Its inputs are plain arrays (tree, page tables, pools,
queries) produced by the seeded generators in ``synth``.

Modules
  tree       -- the query<->node index (KV-guided grouping), the page walk,
                per-query visible token sets and the unique/flat KV byte counts.
  attention  -- decode attention by its definition, the per-node partial
                attention with its stabilised accumulators, and the two-way
                partial-output merge (POR).

Pins (tests/test_oracle_pins.py) tie each function to something other than
itself: brute-force flat attention on sequences materialised from the
generator's logical node arrays, closed forms, merge associativity and
commutativity, the FlashAttention online-softmax loop, and the worked integer
examples printed in the shared-prefix techniques blog.
"""
from . import tree, attention  # noqa: F401
