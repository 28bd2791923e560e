"""Float64 CPU oracle (test infrastructure only; see sinkkv_oracle's header).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference leg
import this package.  The CUDA library never does.
"""
from .sinkkv_oracle import *  # noqa: F401,F403
