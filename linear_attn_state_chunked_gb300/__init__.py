"""GB300-native linear-attention hot path of position-independent caching.

``hypic`` is the ctypes binding of the C-ABI CUDA library (libhypic.so, built
in-tree by ``build_ext``); ``workloads`` draws the seeded synthetic inputs.
The library is loaded on first use and never replaced by a fallback.
"""
from . import hypic, workloads  # noqa: F401
