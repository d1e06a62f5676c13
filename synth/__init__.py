"""Seeded synthetic inputs shared by the oracle and the CUDA path (no method arithmetic)."""
from . import philox, recipes  # noqa: F401
