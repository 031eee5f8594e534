"""Oracle: plain, slow, obviously correct CPU restatements of what the GEMM
library computes.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
CPU-baseline / reference legs of bench.py may import, call or execute anything
in this package.  It shares no code with the product package (no headers, no
helpers, no constants); the two meet only in the seeded input generators.

  oracle.gemm       fp64 GEMM + epilogue (C source gemm_ref.c, built with gcc),
                    bf16 round-to-nearest-even, the normalised error metric.
  oracle.selection  the pages' enumerator, wave arithmetic, workshop model,
                    square-tile traffic law; the GB300 feasibility rules,
                    candidate generator, cost model and tile schedule restated
                    from their documented definitions; rank agreement.

Parity pins (tests/test_oracle_*.py):
  gemm            hand brute force (≤ 3×5×7), identity and permutation matrices,
                  exact integer sums, GELU closed-form points.
  p1_candidates   the printed 12,288-element cap, rule-by-rule brute force.
  workshop        the printed results of "Compilers and Kernel Languages".
  traffic law     explicit tile-loop count = 2N³/T; √(C/3).
  waves           133 tiles on 132 SMs → 2 waves; 64 tiles < half a wave.
  rank agreement  hand cases, and scipy.stats on random data.
  gb300_model     panel bytes = the per-block traffic law summed over tiles;
                  waves and wave efficiency = a round-by-round dispatch of the
                  CTAs; never below the roofline floor; HBM bytes = compulsory
                  bytes when A and B fit in half of L2 (each pin with a planted
                  mistake it catches).  Fitted coefficients: "parity unpinned".
  gb300_candidates  = a brute-force filter of the documented grid; holds the
                  fixed tile.  gb300_check (TMEM/tcgen05 rules): "parity
                  unpinned" against the pages, which say nothing about them;
                  brute force and set-equality with the library only.
  mx, fp8         the OCP format tables, reduction to the plain GEMM oracle,
                  power-of-two invariances, NaN propagation.
"""
from . import gemm, selection  # noqa: F401

__all__ = ["gemm", "selection"]
