"""CPU float64 oracle for R-SWA: test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library.
"""
from .rswa_oracle import *  # noqa: F401,F403
from .rswa_oracle import __all__  # noqa: F401
