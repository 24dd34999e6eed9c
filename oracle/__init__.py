"""CPU oracle (test infrastructure only; see masw_oracle's header)."""
from .masw_oracle import *  # noqa: F401,F403
