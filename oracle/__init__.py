"""Oracle (test infrastructure only): a plain CPU restatement of the hot path.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The library never does.
"""
from .dhs_oracle import *  # noqa: F401,F403
from .dhs_oracle import Config, Oracle, Stats  # noqa: F401
