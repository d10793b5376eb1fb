"""CPU oracle for the DFlash2 draft tail — test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it, and it
never calls the CUDA library.
"""
from .dflash2_oracle import *  # noqa: F401,F403
from . import dflash2_oracle as core  # noqa: F401
