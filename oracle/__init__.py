"""Float64 CPU oracle of the ESM-2 packed encoder forward (test infrastructure only)."""
from .esm_oracle import *  # noqa: F401,F403
