"""Routed mixture-of-experts FFN layer on one B300 (sm_103a).

Submodules:
  capi    -- thin ctypes binding of the C ABI (include/moe.h, include/moe_gen.h); importing it
             fails loudly if the CUDA library libmoe_b300.so has not been built.
  inputs  -- seeded synthetic inputs (no MoE arithmetic).
  build   -- compiles the CUDA library in-tree for sm_103a.
"""
