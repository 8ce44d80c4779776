"""Plain CPU oracle for vertical-slash sparse attention (test infrastructure).

ONLY ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never calls it.
See ``oracle/vs_oracle.py`` (the VS method) and ``oracle/xattn_oracle.py``
(the anti-diagonal block scorer) for the functions and the passages they
follow.
"""
from .vs_oracle import *  # noqa: F401,F403
from .xattn_oracle import *  # noqa: F401,F403
