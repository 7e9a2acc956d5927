"""Paged MoE experts for GB300: K-slot table in HBM, all experts in pinned host memory.

The compute path is libpe.so (CUDA kernels for sm_103a behind a C ABI, see
include/pe.h); ``PagedMoE`` is its thin ctypes binding.  ``synth`` holds the
seeded input generators.  Importing this package does not load the library;
the first ``PagedMoE`` (or ``lib()``) does, and fails loudly if it is missing.
"""

from .synth import MoEShape  # noqa: F401


def __getattr__(name):
    if name in ("PagedMoE", "PEError", "lib", "required_device_bytes", "row_layout", "max_waves"):
        from . import _lib

        return getattr(_lib, name)
    raise AttributeError(name)
