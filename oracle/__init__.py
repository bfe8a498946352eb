"""FP64 CPU oracle (test infrastructure only; see oracle/oracle.py)."""
from .oracle import *  # noqa: F401,F403
from .oracle import ARCHS, Layer, build_layers  # noqa: F401
