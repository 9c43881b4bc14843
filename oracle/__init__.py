"""CPU oracle (test infrastructure only): see oracle/nvfp4_moe.py."""
from .nvfp4_moe import *  # noqa: F401,F403
