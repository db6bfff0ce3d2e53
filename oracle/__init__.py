"""CPU oracle package (test infrastructure; never on the product path)."""
from .jetfp8_oracle import *  # noqa: F401,F403
