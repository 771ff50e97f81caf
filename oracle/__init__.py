"""CPU float64 oracle for Skiparse attention (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and reference
legs may import this package. The product library never does.
"""
from .skiparse_oracle import *  # noqa: F401,F403
from . import skiparse_oracle  # noqa: F401
