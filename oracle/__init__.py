"""CPU fp64 oracle (test infrastructure only; see fia_oracle.py)."""
from . import fia_oracle  # noqa: F401
