"""Float64 CPU oracle — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never imports, links or calls it, and it never imports the library;
the two share only the seeded input generator module.

Every function is pinned by a ``-m "not gpu"`` test (tests/test_oracle_pins.py)
to values fixed by the pages or by mathematics rather than to itself.
"""
from . import bsa_oracle  # noqa: F401
from .bsa_oracle import *  # noqa: F401,F403
