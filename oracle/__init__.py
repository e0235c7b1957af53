"""CPU oracle of MSA decode over an NVFP4 paged cache.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg, never by the product package.  Plain float64 numpy, one
function per step of the method; shares no code with the CUDA path.
"""
from . import cache, formats, msa  # noqa: F401
