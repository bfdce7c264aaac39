"""CPU oracle (test infrastructure only; see wq_oracle's docstring)."""
from .wq_oracle import *  # noqa: F401,F403
