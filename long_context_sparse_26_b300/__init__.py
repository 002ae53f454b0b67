"""DSA sparse attention with IndexShare for B300 (sm_103a).

The compute path is libdsa.so (hand-written CUDA behind a C ABI, see
include/dsa.h); `binding` is its thin ctypes wrapper and `workloads` draws the
seeded synthetic inputs.  Importing this package loads nothing: the library
is opened on first use and every call raises if it is missing.
"""
