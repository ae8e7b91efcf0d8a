"""GB300-native MXFP4 latent-MoE layer (sm_103a).

The layer routes each latent token to k of E experts by sigmoid score, runs
each expert's gate/up projection, SwiGLU and down projection with MXFP4
weights and MXFP8 activations on tcgen05 block-scaled tensor cores, and ends
with the routing-weighted combine to bf16.

Submodules:
  abi    -- ctypes binding of the C-ABI library libmoe.so (same names as
            include/moe.h); loads the library lazily and fails loudly when it
            is missing.
  synth  -- seeded synthetic inputs (no layer arithmetic).
  build  -- compiles libmoe.so for sm_103a.
"""
