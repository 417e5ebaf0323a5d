"""CPU oracle (test infrastructure only; see fp8_oracle.py)."""
from .fp8_oracle import *  # noqa: F401,F403
