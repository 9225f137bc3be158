"""CPU oracle for absorbed MLA decode (test infrastructure only; see mla_oracle)."""
from .mla_oracle import *  # noqa: F401,F403
from . import mla_oracle  # noqa: F401
