"""CPU oracle (test infrastructure only; never imported by the library)."""
from .oracle import *  # noqa: F401,F403
