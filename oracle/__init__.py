"""fp64 CPU oracle of GPTQ's per-layer quantization path (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline / reference arm of
``bench.py`` may import this package.  The CUDA library never does.
"""
from .gptq_oracle import *  # noqa: F401,F403
from .gptq_oracle import __all__  # noqa: F401
