"""fp64 CPU oracle for the Gated DeltaNet recurrence and the layer steps around it.

Test infrastructure: only the test suite, the smoke check and the CPU-baseline
leg of the benchmark use this package.  The library never imports it.
"""
from .oracle import build, recurrence, recurrence_head, library_path  # noqa: F401
from . import layer  # noqa: F401
