"""CPU oracle of the MiniMax-H3 block forward.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are its only callers.  The CUDA library never imports,
links or runs anything here.  See h3_oracle.py for what each function follows.
"""
from .h3_oracle import *  # noqa: F401,F403
from . import h3_oracle  # noqa: F401
