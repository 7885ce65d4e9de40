"""CPU fp64 oracles for dynamic block-sparse attention and for 3D deformable sliding attention.  Test
infrastructure only: the library never imports them."""
from .sda_oracle import *  # noqa: F401,F403
from .sda_oracle import Geometry  # noqa: F401
from . import dsa3d_oracle  # noqa: F401
