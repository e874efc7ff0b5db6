"""CPU oracle for the DiT hot path: test infrastructure, never product code.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline legs may
import this package.
"""
from . import dit_oracle  # noqa: F401
