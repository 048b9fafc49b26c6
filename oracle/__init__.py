"""CPU oracle of the DSA lightning-indexer hot path (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg and
reference arm may import this package.  The CUDA library never uses it.
"""
from .dsa_oracle import *  # noqa: F401,F403
