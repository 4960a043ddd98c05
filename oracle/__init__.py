"""CPU oracle for the DFlash block-draft hot path (test infrastructure only).

Imported by the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg, never by the library or its binding.
"""
from .dflash_oracle import *  # noqa: F401,F403
from . import dflash_oracle  # noqa: F401
