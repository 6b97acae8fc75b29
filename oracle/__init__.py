"""fp64 CPU oracle of the two-stage draft LM head (test infrastructure only;
see lmhead_oracle for its sources and readings)."""
from .lmhead_oracle import *  # noqa: F401,F403
from .lmhead_oracle import fsum_dot  # noqa: F401
