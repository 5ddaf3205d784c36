"""Test infrastructure: the fp64 CPU oracle of the INSTANT low-rank backward.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the C-ABI library and
its Python binding) never calls it and shares no code with it.
"""

from .instant_oracle import *  # noqa: F401,F403
