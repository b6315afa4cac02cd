"""fp64 CPU oracle for exact attention (test infrastructure only).

Only the test suite, the package entry point's smoke check and the benchmark's
CPU-baseline leg may import this package. The CUDA path does not use it.
"""
from . import attn_ref  # noqa: F401
