"""CPU oracle (test infrastructure only; see nm_oracle's module docstring)."""
from .nm_oracle import *  # noqa: F401,F403
