"""fp64 CPU oracle (test infrastructure only; see oracle/reference.py)."""
from .reference import *  # noqa: F401,F403
