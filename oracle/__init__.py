"""Plain fp64 CPU oracle for the Q4_0 decode-step product (test infrastructure).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
use this package.  The GPU library never imports, links or calls it.
"""
from .oracle import *  # noqa: F401,F403
