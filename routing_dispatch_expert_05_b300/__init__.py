"""B300-native sparse Mixture-of-Experts FFN forward.

``moe``        -- ctypes binding of the C ABI (include/moe.h)
``workloads``  -- seeded synthetic workloads (shapes and input draws)
``build``      -- in-tree nvcc build of libmoe_b300.so for sm_103a
"""
from . import workloads  # noqa: F401

__all__ = ["workloads", "moe", "build"]
