"""Test infrastructure: the fp64 CPU oracle (see dsa_oracle.py). Never imported by the product path."""
from .dsa_oracle import *  # noqa: F401,F403
