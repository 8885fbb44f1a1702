"""CPU oracle for the block-scaled quantization hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously-correct
restatement of what the method computes, written in float64 numpy (float32
only where the method itself fixes float32 arithmetic).  It shares no code
with the CUDA path and imports nothing from it.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and its
``--impl reference`` arm) may import it; the product path never does.

Sources restated here (cited by title and section in each function):

* "UE8M0 FP8 / MXFP8 explainer" (ag-981.com news article on UE8M0 FP8 scales):
  section 1 (what UE8M0 / FP8 / MXFP8 are), section 2 (numeric and hardware
  problems solved), section 4 (relation to conventional FP8) and the gap
  section 1 (numerics: floor versus ceil scale rounding) and gap section 2
  (operators: dual row/column copies).
* AstrAI ``astrai/extension/ops/fp8.py`` at commit 962c10c52b: the commit
  message (in-kernel delayed-scaling fold, dual/transposed byte equality) and
  the docstrings of ``quantize`` / ``quantize_dual``.
* "Format-aware fusion for FP4" (theaicronicle.com): the MXFP4 recipe with
  row-gradient stochastic rounding and fixed-sign 32-point Hadamard.
* Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
  (SC'11), section 3.3: the Philox-4x32 bijection.

Functions with no independent pin say "parity unpinned" in their docstring.
"""

from . import formats, philox, mx, pertensor, gemm  # noqa: F401
