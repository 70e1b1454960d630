"""GB300 (sm_103a) BF16 MoE grouped GEMM backward: fused dGLU dgrad and grouped wgrad.

The compute path is the C-ABI library ``libmgg.so`` built from ``csrc/`` (see
``include/mgg.h``); this package is its thin Python binding.  Importing the
package does not load the library; the first call does, and fails loudly if
the library is missing.
"""
__all__ = ["synth"]
