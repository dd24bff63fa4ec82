"""CPU oracle for the MXFP4 grouped MoE path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use this package.  The CUDA library never imports, links or
calls it, and it shares no code with the library.
"""
from .oracle import *  # noqa: F401,F403
