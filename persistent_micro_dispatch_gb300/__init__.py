"""GB300-native persistent micro-op dispatcher (GPUOS hot path).

The C ABI lives in ``libgpuos.so`` (include/gpuos.h); ``gpuos`` is its thin
ctypes binding. Importing this package does not load CUDA; the library is
loaded on first use and its absence is an error, never a fallback.
"""
from . import gpuos  # noqa: F401
from .gpuos import Executor, eager_run, default_config, DESC_DTYPE, OP  # noqa: F401

__all__ = ["gpuos", "Executor", "eager_run", "default_config", "DESC_DTYPE", "OP"]
