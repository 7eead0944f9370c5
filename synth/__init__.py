"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This package draws random numbers and builds per-position cos/sin tables, which
are caller-supplied inputs of the attention step. It holds none of the method's
arithmetic: no rotation, no masking, no attention, no cache bookkeeping.
"""
from .workloads import *  # noqa: F401,F403
