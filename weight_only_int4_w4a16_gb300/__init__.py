"""GB300 (sm_103a) group-wise INT4 weight-only linear layer (W4A16).

The computation lives in the CUDA library built from ``csrc/`` (C ABI in
``include/w4a16.h``); this package is its Python binding.  Import fails if the
library has not been built (``python weight_only_int4_w4a16_gb300/build.py``).
"""
from .binding import *  # noqa: F401,F403
from .binding import (LIB_PATH, LinearDesc, RoundGraph, W4A16Error, lib, make_descs,  # noqa: F401
                      rung_name)
