"""CPU oracle for the BF16 MoE grouped GEMM backward (dGLU / dsReLU dgrad + grouped wgrad).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or link
anything under ``oracle/``; the only callers are ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline`` / ``--impl
reference`` legs.  The oracle shares no code with the CUDA path.

It is a plain, slow, obviously-correct restatement of what the two pages
define, in float64 unless the pages fix the precision:

* "Grouped GEMM + dGLU (SM100)", BF16 contract, "Tensors, layouts, and
  equation": R_g = alpha_g^2 A_g B_g^T, X_g = beta_g C_g, the dSwiGLU and dGeGLU
  derivatives on alternating 32-wide gate/input blocks, the dprob row sum and the
  per-expert dbias, the dSiTU-GLU derivatives of the block-scaled "Equations", and the
  per-expert amax of 16-bit D_row.
* "Grouped GEMM + dsReLU (SM100)", "Equations": D_row = prob * 2 * C * relu(alpha_g A_g B_g^T),
  dprob = sum C * relu(.)^2, the per-expert Amax of 16-bit D_row.
* "Grouped GEMM + WGrad (Unified)", "Operation": Wgrad[e] = A[:, begin:end] @
  B[begin:end, :], overwrite or accumulate_on_output.

Every function is pinned by ``tests/test_oracle_pins.py`` (brute force on tiny
inputs, finite differences, invariants, special cases).  No function is
"parity unpinned".
"""
from .mgg_oracle import *  # noqa: F401,F403
