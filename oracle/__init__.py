"""CPU oracle of the decode hot path -- test infrastructure only (see spc_oracle)."""
from .spc_oracle import *  # noqa: F401,F403
