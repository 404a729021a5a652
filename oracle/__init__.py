"""fp64 CPU oracle of the FAST-AR per-chunk attention path.

Test infrastructure only: imported by the tests, by __graft_entry__.smoke()
and by the CPU-baseline leg of bench.py, never by the library.
"""
from .fastar_oracle import *  # noqa: F401,F403
from .fastar_oracle import CacheState, CapacityError  # noqa: F401
