"""CPU oracle for split-KV decode attention.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check in
``__graft_entry__`` and by the CPU-baseline leg of ``bench.py``; never by the
CUDA library or its Python binding.  See ``fd_oracle`` for what it computes.
"""

from .fd_oracle import *  # noqa: F401,F403
from .fd_oracle import __all__  # noqa: F401
