"""CPU fp64 oracle for dynamic block-sparse attention.  Test infrastructure only: the library never imports it."""
from .sda_oracle import *  # noqa: F401,F403
from .sda_oracle import Geometry  # noqa: F401
