"""CPU oracle for the DFlash block-draft pass: test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
reference legs may import this package.  The product path (the CUDA library
and its Python binding) never imports it and has no CPU fallback.
"""
from .dflash_oracle import *  # noqa: F401,F403
