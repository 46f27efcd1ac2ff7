"""W4A16 NVFP4 mixture-of-experts FFN layer for NVIDIA GB300 (sm_103a).

The C ABI lives in include/moe_w4a16.h and libmoe_w4a16.so (built by
moe_layer_bit_gb300.build); this package holds the ctypes binding (_lib), a
small convenience layer (layer) and the seeded synthetic workloads (workloads).
"""
from . import workloads  # noqa: F401

__all__ = ["workloads"]
