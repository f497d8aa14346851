"""fp64 CPU oracle for the LRMoE backward-recalibration path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only the tests, the smoke check and the bench's CPU
baseline leg use it.  It shares no code with the CUDA library.
"""

from .lrm_oracle import *  # noqa: F401,F403
