"""fp64 CPU oracle for the Llama pre-norm decoder block -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never calls it and shares no code with it; the only module
both sides use is ``synth`` (seeded input draws, no block arithmetic).

Everything here is plain numpy in float64: a matmul (``@``) is the only library
primitive used as a step.  Each function names the page and section of the
method description it restates.  Parity status per function is listed in the
module docstring of :mod:`oracle.llama_block`.
"""
from .llama_block import *  # noqa: F401,F403
