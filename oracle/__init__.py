"""fp64 CPU oracle of the Locks decode hot path (test infrastructure only).

Only the tests, the package smoke check and the bench's CPU-baseline arm may
import this package; the product path never does.
"""
from .locks_oracle import *  # noqa: F401,F403
