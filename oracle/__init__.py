"""CPU oracle for the fp9 FFN/MoE decode step.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, obviously correct
restatement of what the GPU path computes, in float64 numpy. Only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import it. The product path (the CUDA library and its Python
binding) never imports, calls or links anything here, and nothing here
imports the product path.
"""

from .fp9_oracle import *  # noqa: F401,F403
