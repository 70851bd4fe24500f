"""CPU oracle (test infrastructure only; see specdec_oracle's header)."""
from .specdec_oracle import *  # noqa: F401,F403
