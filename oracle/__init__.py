"""fp64 CPU oracle for one Medusa draft-and-verify step.

Test infrastructure only: imported by the tests, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the CUDA library.
"""
from .medusa_oracle import *  # noqa: F401,F403
from . import medusa_oracle  # noqa: F401
