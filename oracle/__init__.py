"""CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does: the CUDA
library has no CPU fallback.
"""

from .hs_oracle import *  # noqa: F401,F403
