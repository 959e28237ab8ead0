"""Float64 CPU oracle (test infrastructure only; never on the product path)."""
from .kv2 import *  # noqa: F401,F403
from . import kv2  # noqa: F401
