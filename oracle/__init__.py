"""CPU oracle of the Gated DeltaNet core (test infrastructure; see core.py)."""
from .core import *  # noqa: F401,F403
from .core import build_oracle  # noqa: F401
