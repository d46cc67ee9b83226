"""CPU oracle for absorbed MLA decode (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library.
"""
from .mla_oracle import *  # noqa: F401,F403
from .workload import *  # noqa: F401,F403
