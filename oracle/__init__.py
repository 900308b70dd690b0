"""Oracle: a plain, slow, obviously correct CPU statement of the suffix prefill.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the
CUDA library (``prefix_reused_prefill_gb300``): not a kernel, header, helper,
table or constant generator.  The only module both sides read is the seeded
input generator ``workloads``.

What it computes (sources are the three pages the design cites):

* ``slots``  -- the slot table's policy: longest-token-prefix match, the
  threshold against the prefix a slot shares with the other slots, empty-slot-
  then-LRU eviction, truncate to the common length, reused-token count
  (goinfer, "Turn nine in under half a second": "How it works").
* ``formats`` -- decoding of the int4 group-32 weight bytes and of bf16 values,
  written from the layout statement in ``include/kvr.h``.
* ``model``  -- the decoder layer stack evaluated row by row: RMSNorm, Q/K/V
  projections, rotate-half RoPE at absolute slot positions, bf16 K/V stored in
  the slot, causal grouped-query attention over the cached prefix plus the new
  rows, O projection, SwiGLU FFN.  A prompt prefilled whole equals its cached
  prefix plus its suffix (goinfer, "What goinfer does"; OpenJev "Accuracy":
  splitting changes only summation order).  The speculative verify of the
  spec-decode post ("cost model") is the same computation for m = k+1 rows;
  the multi-question priming of OpenJev ("What changed") is the same
  computation where each question sees the shared state plus its own rows.

Arithmetic is float64.  Values are rounded to bf16 exactly where the model
stores a bf16 tensor (``numerics.round_bf16``); these rounding points are a
reading of the pages, listed in the design notes.

Parity status of each function is stated in its module header.
"""
