"""Plain fp64 CPU oracle of the Compass-style decoder stack.

TEST INFRASTRUCTURE ONLY: imported by the tests, the package smoke check and the
bench's CPU-baseline leg, never by the library. It shares no code with the CUDA path.
"""
from .decoder import *  # noqa: F401,F403
from . import decoder  # noqa: F401
from . import runs  # noqa: F401,E402
