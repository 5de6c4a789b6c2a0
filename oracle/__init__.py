"""CPU fp64 oracle (test infrastructure only; see hstu_oracle)."""
from .hstu_oracle import *  # noqa: F401,F403
