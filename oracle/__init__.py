"""fp64 CPU oracle (test infrastructure only; see hsa_oracle's header)."""
from .hsa_oracle import *  # noqa: F401,F403
from . import hsa_oracle  # noqa: F401
