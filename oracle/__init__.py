"""CPU oracle (test infrastructure only; never imported by the product path)."""
from .kvq_oracle import *  # noqa: F401,F403
from .kvq_oracle import OracleCache, KIND_K, KIND_V, T, D, TILE  # noqa: F401
