"""Plain, slow CPU oracle for the TetraJet-v2 NVFP4 linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code, table or
constant generator with the CUDA library in ``nvfp4_bit_fully_gb300/csrc``.

Sources.  The method is described by four summary pages of arXiv 2510.27527
("TetraJet-v2: Accurate NVFP4 Training for Large Language Models with
Oscillation Suppression and Outlier Control").  Citations below name the
"technical summary" (gist.science nl/es/ja pages, which agree section for
section) by its section: §2.A double-block quantization, §2.B OsciReset,
§2.C OutControl.  Where the pages are silent, the reading taken is stated at
the function that relies on it.

Precision.  Every decision that produces an integer (an E2M1 code, a scale
byte, a stochastic-rounding choice, a reset bit) is taken in IEEE fp32 with
round-to-nearest-even and no fused multiply-add, exactly as the pages' format
(fp32 outer scale) implies; accumulations of products (the GEMMs) are fp64.

Modules
-------
formats   E2M1 grid, E4M3 / UE8M0 scale formats
philox    Philox4x32-10 counter-based generator (Salmon et al., SC'11)
quant     double-block NVFP4 quantization (RTN / SR), MXFP8 outlier slice
rht       128-point random Hadamard transform
linear    forward / backward (dX, dW) compositions, fp64 GEMM
osci      OsciReset oscillation tracking and reset
calib     OutControl static outlier calibration

Parity status: every function is pinned by a test in ``tests/test_oracle_*.py``
against something other than itself (published known-answer vectors, library
routines, closed forms, brute force, exhaustive enumeration).
"""
