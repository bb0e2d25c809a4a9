"""CPU oracle for the fused weight-gradient + optimizer step.

Test infrastructure only: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library itself.
"""

from .forge_oracle import *  # noqa: F401,F403
from .forge_oracle import Hyper, State, step, step_values  # noqa: F401
