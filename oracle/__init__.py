"""CPU oracle for the NVFP4 path: test infrastructure, never used by the library."""
from .nvfp4_oracle import *  # noqa: F401,F403
