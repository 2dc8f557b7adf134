"""fp64 CPU oracle of the KDA gated delta rule (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import
this package.  It shares no code with the CUDA library.
"""
from .kda_oracle import *  # noqa: F401,F403
