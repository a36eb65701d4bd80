"""CPU oracle for the MoE grouped GEMM: TEST INFRASTRUCTURE, not product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or run anything in this
package.  The CUDA library never calls it, and it shares no code, header,
table or helper with the CUDA path: it is written from the pages alone.

What it computes, and where each rule comes from:

* ``plan``      -- token-tile padding accounting.  Padded token rows
  ``P = sum_i q*ceil(t_i/q)``, useful rows ``U = sum_i t_i``, padding
  fraction ``(P-U)/P`` ("MoE GroupGEMM padding under expert skew",
  "Calculate padded token columns"), effective experts ``U^2 / sum t_i^2``
  (same page, "Summarize skew without losing the histogram"), per-expert
  segment offsets aligned to the token block ("flops/deepgemm-grouped-masked-
  moe-gemm", "Arithmetic intensity": each expert segment aligned to the GEMM
  M block), the tile list, and the single-GEMM M-occupancy of "Query on
  performance-modeling of MoE Grouped GEMM", "Background".
* ``numerics``  -- decoders for the operand encodings: bf16, FP8 E4M3 and
  UE8M0 power-of-two scale bytes ("flops/deepgemm-grouped-masked-moe-gemm",
  "Workarounds": FP8 with per-group scaling, UE8M0 on SM100), plus the
  block-scale dequantisation of activations (one scale per row and 128 K)
  and weights (one scale per 128 N x 128 K block); E2M1 4-bit weights with
  one UE8M0 scale per (row, 32 K) (same section: FP8 x FP4 MoE GEMMs).
* ``gemm``      -- the three grouped GEMM forms, in float64 on dequantised
  inputs: M-grouped contiguous, masked, and K-grouped weight gradient
  ("flops/deepgemm-grouped-masked-moe-gemm", "Arithmetic intensity" and
  "Workarounds"; "MoE GroupGEMM padding under expert skew", "Grouped execution
  does not require padded experts").
* ``epilogue``  -- SwiGLU of GEMM1's gate and up halves and the E4M3 / UE8M0
  re-quantisation that feeds GEMM2 ("flops/deepgemm-grouped-masked-moe-gemm",
  "Workarounds": SwiGLU fused between the two grouped GEMMs of the MoE).
* ``selector``  -- the exemplar choice of a token tile from the count
  histogram ("MoE GroupGEMM padding under expert skew", "Adapt kernels
  without adding a CPU stall"), in integers.

Every function is pinned by ``tests/test_oracle_*.py`` against values the
pages print, closed forms, invariants and brute force; no function here is
"parity unpinned".
"""

from . import plan, numerics, gemm, epilogue, selector  # noqa: F401
