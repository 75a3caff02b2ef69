"""fp64 CPU oracle for exact attention (test infrastructure).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package. The CUDA library never does, and this package never
imports the CUDA library.
"""
from .naive import attention, attention_head, attention_rows, to_f64  # noqa: F401
