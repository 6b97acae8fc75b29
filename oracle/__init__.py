"""fp64 CPU oracle of the two-stage draft LM head and of the steps that
consume its q (test infrastructure only; see lmhead_oracle and
speculative_oracle for their sources and readings)."""
from .lmhead_oracle import *  # noqa: F401,F403
from .lmhead_oracle import fsum_dot  # noqa: F401
from .speculative_oracle import *  # noqa: F401,F403
