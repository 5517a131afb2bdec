"""CPU oracle for the context-parallel ring-attention step.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, fp64 NumPy
restatement of what the pages define. Only the tests, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The CUDA library never calls it, and it shares no code with the CUDA path:
the only common module is ``workloads`` (seeded random inputs).

``oracle.fp8`` holds the E4M3 format and the per-tensor FP8 quantization of
the FP8 path; its attention is ``attention`` on the dequantized values.

Parity status per function (see the pins in ``tests/test_oracle_*.py``):
every public function here is pinned against something other than itself
(a worked example printed on the pages, closed forms, brute force on tiny
inputs, invariants, a library special case, finite differences).
"""
from .ring_attention import *  # noqa: F401,F403
from .ring_attention import __all__  # noqa: F401
