"""fp64 CPU oracle of ResidualQuant (test infrastructure only; see rq_oracle)."""

from .rq_oracle import *  # noqa: F401,F403
from .rq_oracle import GROUP  # noqa: F401
