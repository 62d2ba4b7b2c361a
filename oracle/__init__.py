"""Oracle package: float64 CPU restatement of the fused path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product path never does.
"""
from .cf_oracle import *  # noqa: F401,F403
from .cf_oracle import __all__  # noqa: F401
