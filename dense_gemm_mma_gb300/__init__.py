"""GB300-native dense GEMM / GEMV library (sm_103a).

The compute path lives in ``libdgemm_gb300.so`` (``csrc/``), a C-ABI shared
library; ``gemm`` is its thin ctypes binding.  ``inputs`` draws the seeded
synthetic operands used by the tests and the benchmark.
"""
