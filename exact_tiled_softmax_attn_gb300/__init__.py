"""Exact tiled softmax attention on NVIDIA GB300 (sm_103a).

The compute lives in libattn.so (C ABI: include/attn.h), built from
``csrc/`` with ``python -m exact_tiled_softmax_attn_gb300.build``. This
package holds the ctypes binding (``binding``), the build step (``build``)
and the seeded workload generator (``workloads``).
"""
from .binding import *  # noqa: F401,F403
from .binding import __all__ as _binding_all

__all__ = list(_binding_all)
