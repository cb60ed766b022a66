"""Order-independent floating-point summation on one GB300 (sm_103a).

The compute path is the C-ABI library built from `csrc/` (see
`include/repro.h`); `api` is its thin ctypes binding.  Importing this package
does not load the library: `api` loads it on first use and raises if it is
missing, with no CPU fallback.
"""
