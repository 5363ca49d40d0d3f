"""CPU oracle (test infrastructure only; never imported by the product path)."""
from .cacheblend_oracle import *  # noqa: F401,F403
