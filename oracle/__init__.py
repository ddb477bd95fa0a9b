"""CPU oracle of the routed MoE layer with an LRU expert-slot cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, links or executes this
package; only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` do.  It shares no code with the CUDA path: the two meet only in the seeded
input generator ``ft_synth``.

* ``oracle.moe``  - router logits in a fixed fp32 order, top-k, renormalised softmax gates,
  the permutation grouped by expert, the SwiGLU expert FFN and the weighted combine
  (fp64), and an independently written dense SwiGLU FFN for the 1-expert special case.
* ``oracle.lru``  - the slot-level LRU cache simulator (slot table, owners, stamps, fills,
  resize, optional frequency admission) and an independently written brute-force LRU used
  to pin it.
* ``oracle.fp4``  - MXFP4 entries: E2M1 codes and E8M0 block scales dequantized exactly, and
  the SwiGLU expert on the dequantized weights.

Sources.  The system is FreeToken as described on the freetoken.wiki pages
"FreeToken RTX 4090" (section "how the MoE memory hierarchy works": complete
layer-expert cache entries, one logical mapping, a shared LRU across layers and tokens),
"FreeToken benchmark" (section "how FreeToken serves large MoE models": host-resident
expert pool, elastic GPU cache, full-layer double buffering in prefill, shared LRU in
decode) and "FreeToken vram" (elastic cache rebuilt at scheduler safe points).  The pages
give no router formula, gate normalisation, FFN form, permutation order or LRU
tie-breaks; each function states the reading it implements.

Every function here is pinned by tests against something other than itself
(brute force, closed forms, hand-derived golden values, library routines for special
cases); see ``tests/test_oracle_*.py``.  No function is "parity unpinned".
"""
