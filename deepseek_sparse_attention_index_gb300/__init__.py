"""DeepSeek Sparse Attention forward hot path for GB300 (sm_103a).

The compute lives in the CUDA library ``libdsa_gb300.so`` (C ABI declared in
include/dsa.h).  ``ops`` is the thin ctypes binding over it; ``inputs`` makes
seeded synthetic workloads.  Importing the package does not load the library;
the first call into ``ops`` does, and fails loudly if it is missing.
"""
