"""fp64 CPU oracle for absorbed MLA decode (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
import this package.  It shares no code with the CUDA path.
"""
from .mla_oracle import *  # noqa: F401,F403
from .workload import *  # noqa: F401,F403
