"""FP64 CPU oracle (test infrastructure only; see kvgqa_oracle.py)."""
from .kvgqa_oracle import *  # noqa: F401,F403
from . import kvgqa_oracle  # noqa: F401
