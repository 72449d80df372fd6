"""B300-native (sm_103a) DeepSeekMoE layer forward.

The compute lives in a C-ABI shared library of hand-written CUDA kernels
(``libmoe_b300.so``, declared in ``include/moe_b300.h``); this package holds
its thin ctypes binding, the named workload shapes and the seeded input
generator.
"""
from .configs import CONFIGS, MoEConfig  # noqa: F401
