"""CPU oracle (test infrastructure only; see h3_oracle's header)."""
from .h3_oracle import *  # noqa: F401,F403
