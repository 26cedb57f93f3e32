"""CPU oracle for one layer-step of RAG KV-cache fusion (test infrastructure).

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it.
"""

from .fusion import *  # noqa: F401,F403
