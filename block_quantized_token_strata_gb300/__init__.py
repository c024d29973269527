"""Block-quantized multi-token verify path for one GB300 (sm_103a).

The compute path is the C-ABI library ``libstrata.so`` (hand-written CUDA, see ``include/strata.h``);
``block_quantized_token_strata_gb300.strata`` is its thin ctypes binding and ``synth`` the seeded
input generator. Importing the package does not load the library; the first call through the
binding does, and fails loudly if it has not been built.
"""
__all__ = ["synth", "strata"]
