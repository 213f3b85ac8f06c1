"""libnvfp4moe for GB300 (sm_103a): the NVFP4 block-scaled Mixture-of-Experts
expert layer as a C-ABI CUDA library with a thin Python binding.

Submodules:
  binding    ctypes binding of libnvfp4moe.so (fails loudly if not built)
  workloads  seeded synthetic layer inputs
  build      nvcc build of the shared library
"""
import importlib

__all__ = ["binding", "workloads", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
