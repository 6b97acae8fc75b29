"""fp64 CPU oracle of the two-stage draft LM head, of its cluster-level
variant and of the steps that consume its q (test infrastructure only; see
lmhead_oracle, cluster_oracle and speculative_oracle for their sources and
readings)."""
from .lmhead_oracle import *  # noqa: F401,F403
from .lmhead_oracle import fsum_dot  # noqa: F401
from .speculative_oracle import *  # noqa: F401,F403
from .cluster_oracle import *  # noqa: F401,F403
