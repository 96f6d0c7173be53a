"""GB300-native balanced expert-parallel hot path (MoonEP-style).

The library (libmoonep.so, C ABI in include/moonep.h) holds the planner,
fused-permute dispatch, combine, redundant-expert weight prefetch and gradient
reduce as hand-written sm_103a CUDA kernels.  ``api.Buffer`` is the PyTorch
front end; ``_lib`` is the raw ctypes binding; ``workloads`` generates seeded
synthetic inputs.
"""
from . import workloads  # noqa: F401


def load_library():
    """Load libmoonep.so (raises if it has not been built)."""
    from . import _lib
    return _lib.load()


def __getattr__(name):
    if name in ("Buffer", "CommPlan", "BufferPool"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
