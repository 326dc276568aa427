"""CPU oracle for the paged KV cache hot path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.
"""

from .oracle import *  # noqa: F401,F403
from .oracle import __all__  # noqa: F401
