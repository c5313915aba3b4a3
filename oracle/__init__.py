"""CPU oracle (test infrastructure only; see qz_oracle's header)."""
from .qz_oracle import *  # noqa: F401,F403
