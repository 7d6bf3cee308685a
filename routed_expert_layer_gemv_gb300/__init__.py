"""One routed MoE layer forward pass on a GB300 (sm_103a), behind a C ABI.

``capi``      ctypes binding of include/moe.h (the library does all the work)
``layer``     set-up helpers: pack FP4 experts into the host pool, install
``workloads`` seeded synthetic inputs of the measured layer shapes
``build``     compiles libmoe_gb300.so in-tree with nvcc
"""
from . import build, capi, workloads  # noqa: F401
