"""fp64 CPU oracle (test infrastructure only; never imported by the product path)."""
from .attention import *  # noqa: F401,F403
from .attention import __all__  # noqa: F401
