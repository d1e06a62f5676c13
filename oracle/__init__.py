"""fp64 CPU oracle (test infrastructure only; see kfsvd_oracle.py's header)."""
from .kfsvd_oracle import *  # noqa: F401,F403
