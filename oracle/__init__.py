"""CPU oracle for the Orthros attention hot path (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
import this package. The CUDA library never does.
"""
from .orthros_ref import (  # noqa: F401
    Oracle, build, decode, extend, max_threads, prefill, prefill_backward, qkv_project)
