"""Float64 CPU oracle (test infrastructure only; see tsa_oracle's header)."""
from .tsa_oracle import *  # noqa: F401,F403
