"""fp64 CPU oracle for exact attention (test infrastructure, see attention_fp64)."""
from .attention_fp64 import *  # noqa: F401,F403
