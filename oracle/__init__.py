"""fp64 CPU oracle of the POET-X layer and the Cayley-Neumann parameterization.

Test infrastructure only: imported by tests/, __graft_entry__.smoke() and the CPU-baseline
leg of bench.py, never by the product path.
"""
from .poetx_oracle import *  # noqa: F401,F403
