"""fp64 CPU oracle for fused linear cross-entropy (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import this
package. The library itself never calls it and shares no code with it.
"""
from .flce_oracle import *  # noqa: F401,F403
from .flce_oracle import __all__  # noqa: F401
