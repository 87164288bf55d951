"""Routed-expert MoE layer with weight-only NVFP4 (W4A16) experts on GB300,
and the dense W4A16 NVFP4 linear that shares its kernels.

The computation lives in the CUDA library libnvfp4moe.so (C ABI declared in
include/nvfp4_moe.h); this package holds its sources (csrc/), the in-tree
build step (build.py) and a ctypes binding (binding.py).
"""
from .build import build, LIB  # noqa: F401
from . import binding  # noqa: F401
from .binding import (  # noqa: F401
    MoELayer, Linear, Nvfp4MoeError, load_library, header_functions, upload_layer,
    PATH_AUTO, PATH_DECODE, PATH_PREFILL, STATUS, STATUS_CODE,
)
