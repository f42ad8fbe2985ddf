"""B300-native Dynamic Short Convolutions (DSC).

The hot path -- head-wise and low-rank DSC, forward and backward -- is CUDA
for sm_103a in ``libdsc.so`` behind the C ABI declared in ``include/dsc.h``.
``dsc`` is the thin ctypes binding to it; ``synthetic`` draws seeded inputs.
Importing the package loads nothing; the binding loads the library on first
use and raises if it is missing.
"""
__all__ = ["dsc", "synthetic"]
