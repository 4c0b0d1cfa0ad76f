"""CPU oracle of the AdaLN diffusion-transformer block forward, its int8lin variant, the FlowMatch
Euler step and the denoise loop.

TEST INFRASTRUCTURE ONLY. Nothing in the product imports, links or runs anything here; only the
tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and reference legs do. It shares
no code with the CUDA path: its only common dependency is the seeded input generator
``dit_inputs``, which draws random numbers and holds none of the method's arithmetic.

Everything is plain NumPy in float64, except where the pages fix a precision: the Euler update is
float32 (the RGBA-Image-2.1 host contract, section 6, "all arrays are fp32") and the int8lin
dequantised weight is rounded to bfloat16 (same contract, section 1), and the W8A8 quantisers take
their code decisions in float32 with the activation at its bfloat16 value (``w8a8``). Weights enter
as the exact values of their bfloat16 bit patterns; no other intermediate activation is rounded.

Parity status: every function here is pinned by a ``-m "not gpu"`` test in ``tests/test_oracle_*.py``
against closed forms, invariants, brute force on tiny inputs or values the pages print. No function
is "parity unpinned".
"""

from .dit import *  # noqa: F401,F403
from .w8a8 import *  # noqa: F401,F403
