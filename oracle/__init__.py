"""CPU oracle for packed varlen non-causal attention with the fused q/k
prologue (per-head RMSNorm, then 3D rotary embedding on 96 of 128 dims).

TEST INFRASTRUCTURE ONLY.  This package is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``;
nothing in the library path imports, links or calls it, and it imports
nothing from the library.  It is plain, slow, fp64 numpy written from the
definitions on the pages:

* ``oracle.plan``       -- cu_seqlens and the fp64 (t, h, w) position grid;
* ``oracle.prologue``   -- RMSNorm with gain, then NeoX rotate-half rotary on
                           dims 0..95 with angles from the position grid;
* ``oracle.attention``  -- per-document bidirectional softmax attention,
                           evaluated with a two-pass (max, then sum) softmax;
* ``oracle.fp8``        -- the FP8 (e4m3) variant: quantisers, dequantisation
                           and the error bound of the kernel's P rounding.

Pages cited (page title, then section):
  [PR26]   vllm.cpp PR #26 "feat(minimax-h3): port the MiniMax-H3 omni-modal
           video+audio DiT"
  [SPARK]  "h3-spark" model card, "MiniMax H3 -- single DGX Spark (GB10)
           serving package"

Parity status of each function is recorded in its docstring; every function
here is pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle_pins.py``.
"""
from . import plan, prologue, attention  # noqa: F401
